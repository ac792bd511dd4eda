"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.

Bars: layout, slot map, identity metadata, bf16 dispatch rows, FP8 payloads
and scales are bit-exact; combine within 1 bf16 ulp, |d| <= 2^-7 |ref| + 1e-6
(expected bit-exact: both sides fold in fp32 with fmaf in ascending k and
cast once).  Every case is compared element by element, the workloads' full
sizes included: the oracle defines each dispatched row token by token, so its
rows are computed once per token and every copy the GPU wrote is compared
with them.  NaN results compare by NaN-ness (IEEE leaves the sign of an
invalid operation's NaN open, so an E4M3 NaN code may be 0x7F or 0xFF).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_REL = 2.0**-7
TOL_ABS = 1e-6


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import load_build_module

    load_build_module().build()
    import combine_get_layout_gb300 as ep

    return ep


_INPUT_CACHE = {}


def inputs(wl, seed=0):
    key = (wl, seed)
    if key not in _INPUT_CACHE:
        _INPUT_CACHE.clear()
        _INPUT_CACHE[key] = workloads.make_inputs(wl, seed=seed)
    return _INPUT_CACHE[key]


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(u16):
    return dev(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(u16):
    return oracle.bf16_to_f32_array(u16)


def cfg_of(ep, wl, zero_padding=False, max_tokens=None):
    return ep.Config(max_tokens or max(wl.num_tokens, 1), wl.hidden, wl.num_topk,
                     wl.num_experts, wl.num_ranks, wl.expert_alignment,
                     wl.use_fp8_dispatch, zero_padding)


def oracle_layout(wl, idx, cap):
    lay = oracle.layout(idx, wl.num_experts, wl.num_ranks, wl.expert_alignment, cap=cap)
    assert lay["status"] == oracle.OK
    return lay


def assert_layout_equal(L, ora, T):
    assert L.num_tokens == T
    g = lambda t: t.cpu().numpy()
    assert np.array_equal(g(L.expert_count), ora["expert_count"])
    assert np.array_equal(g(L.expert_start), ora["expert_start"])
    assert np.array_equal(g(L.expert_end), ora["expert_end"])
    assert np.array_equal(g(L.rank_start), ora["rank_start"])
    assert np.array_equal(g(L.tokens_per_rank), ora["tokens_per_rank"])
    assert np.array_equal(g(L.is_token_in_rank)[:T], ora["is_token_in_rank"])
    assert np.array_equal(g(L.slot_of)[:T], ora["slot_of"])
    used = int(ora["expert_start"][-1])
    assert np.array_equal(g(L.src_info)[:used], ora["src_info"][:used])
    assert int(g(L.err)[0]) == 0


def assert_combine_close(got_u16, ref_u16):
    g = f32(got_u16).astype(np.float64)
    r = f32(ref_u16).astype(np.float64)
    assert np.all(np.abs(g - r) <= TOL_REL * np.abs(r) + TOL_ABS)


def run_layout(ep, cfg, idx_np, sync=True):
    idx = dev(idx_np)
    L = ep.get_layout(cfg, idx, sync=sync)
    torch.cuda.synchronize()
    return L


# --------------------------------------------------------------------------
# workloads and edge cases
# --------------------------------------------------------------------------

FULL = ["tiny", "decode", "prefill", "skew", "sweep1k", "sweep4k", "sweep16k"]

MEDIUM = {
    # several layout tiles with a ragged last tile, masked slots, small A
    "ragged_bf16": workloads.Workload("ragged_bf16", 1000, 1024, 64, 8, 8, False,
                                      expert_alignment=16, mask_frac=0.07),
    "ragged_fp8": workloads.Workload("ragged_fp8", 333, 1024, 32, 4, 4, True,
                                     expert_alignment=8, mask_frac=0.1),
    "k1_e_eq_r": workloads.Workload("k1_e_eq_r", 257, 256, 16, 1, 16, False,
                                    expert_alignment=1),
    "wide_experts": workloads.Workload("wide_experts", 100, 128, 2048, 32, 64, True,
                                       expert_alignment=4),
    "skew_small": workloads.Workload("skew_small", 700, 512, 64, 6, 8, True,
                                     zipf_alpha=1.2, mask_frac=0.05),
    "many_tiles": workloads.Workload("many_tiles", 70000, 8, 256, 8, 8, False),
    # the largest expert and rank counts: count rows of 4096 entries,
    # streamed two rows at a time; byte-wise rank flags
    "max_experts_ranks": workloads.Workload("max_experts_ranks", 1000, 128, 2048, 8, 2048,
                                            False, expert_alignment=4, mask_frac=0.05),
    # one expert, past the one-launch limit: 8-entry count rows, most row
    # groups of the column sums empty
    "one_expert_big": workloads.Workload("one_expert_big", 5000, 64, 1, 1, 1, False,
                                         expert_alignment=1),
    # 2048 experts over 31 tiles: the tile-count matrix exceeds shared
    # memory and is streamed through the two-buffer ring
    "ring_scan": workloads.Workload("ring_scan", 1000, 128, 2048, 8, 64, False,
                                    expert_alignment=4, mask_frac=0.05),
    # more than 64 destination ranks (byte-wise rank rows), both layout paths
    "wide_ranks_small": workloads.Workload("wide_ranks_small", 100, 128, 256, 8, 128, False,
                                           expert_alignment=4, mask_frac=0.05),
    "wide_ranks": workloads.Workload("wide_ranks", 2000, 128, 256, 8, 128, False,
                                     expert_alignment=4, mask_frac=0.05),
    # either side of the one-launch layout's limit of 4096 (t, k) pairs
    "small_edge": workloads.Workload("small_edge", 512, 256, 64, 8, 8, False,
                                     expert_alignment=16, mask_frac=0.05),
    "past_small_edge": workloads.Workload("past_small_edge", 513, 256, 64, 8, 8, False,
                                          expert_alignment=16, mask_frac=0.05),
}


@pytest.mark.parametrize("name", FULL + list(MEDIUM))
def test_layout_bit_exact(ep, name):
    wl = workloads.WORKLOADS.get(name) or MEDIUM[name]
    inp = inputs(wl)
    cfg = cfg_of(ep, wl)
    L = run_layout(ep, cfg, inp["topk_idx"])
    ora = oracle_layout(wl, inp["topk_idx"], cfg.capacity)
    assert_layout_equal(L, ora, wl.num_tokens)
    assert np.array_equal(L.h_expert_count, ora["expert_count"])


def test_layout_more_tiles_than_target(ep):
    """A token count large enough that tiles hit their maximum size."""
    wl = workloads.Workload("big", 200000, 8, 64, 4, 8, False)
    rng = np.random.default_rng(4)
    idx = workloads.random_routes(rng, wl.num_tokens, wl.num_experts, wl.num_topk, 0.02)
    cfg = cfg_of(ep, wl)
    L = run_layout(ep, cfg, idx)
    assert_layout_equal(L, oracle_layout(wl, idx, cfg.capacity), wl.num_tokens)


@pytest.mark.parametrize("T,K,E,R", [
    # 152 tiles of exactly 65535 pairs, every pair on one expert: each
    # tile's count is the largest a 16-bit count holds
    (152 * 65535, 1, 1, 1),
    # tiles of 68,424 pairs: past 16-bit counts, the 32-bit rows
    (1_300_000, 8, 64, 8),
])
def test_layout_tile_count_width_edges(ep, T, K, E, R):
    wl = workloads.Workload("edge", T, 8, E, K, R, False, expert_alignment=4)
    if E == 1:
        idx = np.zeros((T, 1), np.int64)
    else:
        rng = np.random.default_rng(15)
        idx = np.empty((T, K), np.int64)
        for c0 in range(0, T, 100_000):           # distinct experts per token
            n = min(100_000, T - c0)
            idx[c0:c0 + n] = np.argsort(rng.random((n, E)), axis=1)[:, :K]
    cfg = cfg_of(ep, wl)
    L = run_layout(ep, cfg, idx)
    assert_layout_equal(L, oracle_layout(wl, idx, cfg.capacity), T)


@pytest.mark.parametrize("T", [5000, 1000])
def test_layout_hot_expert(ep, T):
    """Every token picks expert 0 plus others: one expert holds T rows (both
    layout paths: 20000 and 4000 (t, k) pairs)."""
    E, K = 32, 4
    rng = np.random.default_rng(5)
    idx = workloads.random_routes(rng, T, E - 1, K - 1) + 1
    idx = np.concatenate([np.zeros((T, 1), np.int64), idx], axis=1)
    wl = workloads.Workload("hot", T, 64, E, K, 4, False)
    cfg = cfg_of(ep, wl)
    L = run_layout(ep, cfg, idx)
    assert_layout_equal(L, oracle_layout(wl, idx, cfg.capacity), T)


def test_layout_empty_and_all_masked(ep):
    wl = workloads.Workload("e", 64, 128, 8, 2, 2, False, expert_alignment=4)
    cfg = cfg_of(ep, wl)
    L = ep.Layout(cfg)
    ep.get_layout(cfg, torch.zeros((0, 2), dtype=torch.int64, device="cuda"), layout=L, sync=True)
    assert L.num_tokens == 0
    assert int(L.expert_start[-1]) == 0 and int(L.expert_count.sum()) == 0
    idx = np.full((64, 2), -1, np.int64)
    L = run_layout(ep, cfg, idx)
    assert_layout_equal(L, oracle_layout(wl, idx, cfg.capacity), 64)
    # combine of all-masked tokens is +0.0
    y = ep.combine(cfg, L, torch.ones((cfg.capacity, 128), dtype=torch.bfloat16, device="cuda"))
    assert np.all(host_u16(y) == 0)


def test_layout_asynchronous_then_check(ep):
    wl = workloads.WORKLOADS["tiny"]
    inp = inputs(wl)
    cfg = cfg_of(ep, wl)
    L = ep.get_layout(cfg, dev(inp["topk_idx"]), sync=False)
    assert ep.check_error(L) == ep.EP_OK
    assert_layout_equal(L, oracle_layout(wl, inp["topk_idx"], cfg.capacity), wl.num_tokens)


@pytest.mark.parametrize("bad,status", [
    ("range_hi", 2), ("range_lo", 2), ("dup", 3), ("both", 2)])
def test_routing_errors_reported(ep, bad, status):
    wl = workloads.Workload("err", 40, 128, 8, 3, 2, False, expert_alignment=4)
    rng = np.random.default_rng(6)
    idx = workloads.random_routes(rng, 40, 8, 3)
    if bad in ("range_hi", "both"):
        idx[7, 1] = 8
    if bad == "range_lo":
        idx[3, 0] = -5
    if bad in ("dup", "both"):
        idx[20, 2] = idx[20, 0]
    cfg = cfg_of(ep, wl)
    d_idx = dev(idx)
    with pytest.raises(ep.EpError) as ei:
        ep.get_layout(cfg, d_idx, sync=True)
    assert ei.value.status == status
    L = ep.get_layout(cfg, d_idx, sync=False)
    assert ep.check_error(L) == status
    # dispatch / combine on a flagged layout stay in bounds and run
    x = dev_bf16(workloads.to_bf16_bits(rng.standard_normal((40, 128))))
    recv, _, _ = ep.dispatch(cfg, L, x)
    ep.combine(cfg, L, recv)
    torch.cuda.synchronize()
    # the next good layout clears the error word
    good = workloads.random_routes(rng, 40, 8, 3)
    L = ep.get_layout(cfg, dev(good), layout=L, sync=True)
    assert ep.check_error(L) == ep.EP_OK


def test_bounded_wait_times_out_cleanly(ep):
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    st = ep.ep_selftest_wait_timeout(2_000_000, err.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == ep.EP_ERR_TIMEOUT
    assert int(err[0]) == 4
    # the context is still usable
    assert float(torch.ones(3, device="cuda").sum()) == 3.0


def _stream_ptr():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("stall_tile,timeout_ns", [(1, 1000), (77, 1_000_000), (151, 1000)])
def test_layout_own_wait_times_out_and_is_reported(ep, stall_tile, timeout_ns):
    """The two-launch layout's bounded wait, run out in one CTA other than 0:
    with a 1 us limit that CTA records the timeout before CTA 0 publishes the
    routing errors, and the publish keeps it (OR, not a store); with 1 ms it
    records after.  Either way the status is EP_ERR_TIMEOUT, the context stays
    usable, and the next good layout reports EP_OK and is exact."""
    wl = workloads.WORKLOADS["prefill"]          # 128 token tiles, 152 CTAs
    inp = inputs(wl)
    cfg = cfg_of(ep, wl)
    idx = dev(inp["topk_idx"])
    L = ep.Layout(cfg)
    st = ep.ep_selftest_layout_timeout(cfg.c(), wl.num_tokens, idx.data_ptr(), L.c,
                                       stall_tile, timeout_ns, _stream_ptr())
    assert st == ep.EP_ERR_TIMEOUT, ep.ep_status_str(st)
    assert ep.ep_check_error(L.c, _stream_ptr()) == ep.EP_ERR_TIMEOUT
    assert float(torch.ones(3, device="cuda").sum()) == 3.0
    ep.get_layout(cfg, idx, layout=L, sync=True)
    assert ep.check_error(L) == ep.EP_OK
    assert_layout_equal(L, oracle_layout(wl, inp["topk_idx"], cfg.capacity), wl.num_tokens)


def test_layout_timeout_in_cta0_replaces_earlier_status(ep):
    """CTA 0 (the one that publishes) runs out of time after a call that left
    a routing error in the word: the word was cleared at the start of the
    call, so the status is the timeout alone, never the earlier error."""
    wl = workloads.WORKLOADS["skew"]
    inp = inputs(wl)
    cfg = cfg_of(ep, wl)
    bad = inp["topk_idx"].copy()
    bad[5, 1] = wl.num_experts                   # out of range
    L = ep.Layout(cfg)
    ep.get_layout(cfg, dev(bad), layout=L, sync=False)
    assert ep.check_error(L) == ep.EP_ERR_EXPERT_RANGE
    idx = dev(inp["topk_idx"])
    st = ep.ep_selftest_layout_timeout(cfg.c(), wl.num_tokens, idx.data_ptr(), L.c, 0,
                                       1000, _stream_ptr())
    assert st == ep.EP_ERR_TIMEOUT, ep.ep_status_str(st)
    ep.get_layout(cfg, idx, layout=L, sync=True)
    assert ep.check_error(L) == ep.EP_OK
    assert_layout_equal(L, oracle_layout(wl, inp["topk_idx"], cfg.capacity), wl.num_tokens)


# --------------------------------------------------------------------------
# dispatch
# --------------------------------------------------------------------------

def _dispatch_case(ep, wl, zero_padding, seed=0):
    inp = inputs(wl, seed)
    cfg = cfg_of(ep, wl, zero_padding=zero_padding)
    L = run_layout(ep, cfg, inp["topk_idx"])
    x = dev_bf16(inp["x"])
    w = dev(inp["topk_weights"])
    recv_x, recv_s, recv_w = ep.dispatch(cfg, L, x, w)
    torch.cuda.synchronize()
    ora = oracle_layout(wl, inp["topk_idx"], cfg.capacity)
    return inp, cfg, L, ora, recv_x, recv_s, recv_w


@pytest.mark.parametrize("name,zp", [("tiny", False), ("tiny", True),
                                     ("ragged_bf16", True), ("ragged_bf16", False),
                                     ("k1_e_eq_r", True), ("prefill", False),
                                     ("sweep1k", True)])
def test_dispatch_bf16_bit_exact(ep, name, zp):
    wl = workloads.WORKLOADS.get(name) or MEDIUM[name]
    inp, cfg, L, ora, recv_x, _, recv_w = _dispatch_case(ep, wl, zp)
    used = int(ora["expert_start"][-1])
    ref_x, ref_w = oracle.dispatch_bf16(inp["x"], inp["topk_weights"], ora, zero_padding=zp)
    got_x = host_u16(recv_x[:used])
    got_w = recv_w[:used].cpu().numpy()
    rows = ora["src_info"][:used, 0] >= 0
    if zp:
        rows[:] = True
    assert np.array_equal(got_x[rows], ref_x[:used][rows])
    assert np.array_equal(got_w[rows], ref_w[:used][rows])


def _identity_slots(n):
    """A layout of n tokens with one row each (row i = token i)."""
    return {"slot_of": np.arange(n, dtype=np.int32).reshape(-1, 1), "cap": n,
            "expert_start": np.array([0, n], np.int32), "expert_end": np.array([n], np.int32),
            "expert_count": np.array([n], np.int32)}


def _fp8_oracle_rows(x_rows):
    """Oracle quantisation of each given bf16 row (one slot per row)."""
    q, s, _ = oracle.dispatch_fp8(x_rows, None, _identity_slots(x_rows.shape[0]))
    return q, s


def _bf16_oracle_rows(x_rows):
    """Oracle dispatch of each given bf16 row (one slot per row)."""
    r, _ = oracle.dispatch_bf16(x_rows, None, _identity_slots(x_rows.shape[0]))
    return r


def _canon_e4m3(q):
    """E4M3 codes with both NaN codes (S.1111.111) mapped to 0x7F."""
    return torch.where((q & 0x7F) == 0x7F, torch.full_like(q, 0x7F), q)


def assert_rows_equal_oracle(inp, ora, fp8, recv, recv_s=None, recv_w=None,
                             zero_padding=False, chunk=4096):
    """Every row in use against the oracle's rows, element by element.

    The oracle's dispatch defines the row of each unmasked (t, k) from x[t]
    alone, so its rows are computed once per token and compared with every
    copy the GPU wrote (rows slot_of[t, k] for all k).  Weights ride along
    per (t, k); alignment gap rows are all-zero bits when zero_padding."""
    x, w = inp["x"], inp["topk_weights"]
    T = x.shape[0]
    if fp8:
        ref_q, ref_s = _fp8_oracle_rows(x)
        ref = torch.from_numpy(ref_q).cuda()
        ref_sc = torch.from_numpy(ref_s.view(np.int32)).cuda()
        got = recv
        got_sc = recv_s.view(torch.int32)
    else:
        ref = torch.from_numpy(_bf16_oracle_rows(x).view(np.int16)).cuda()
        got = recv.view(torch.int16)
    slot = torch.from_numpy(ora["slot_of"]).cuda().long()
    m = slot >= 0
    tok = torch.arange(T, device="cuda").unsqueeze(1).expand_as(slot)[m]
    kk = torch.arange(slot.shape[1], device="cuda").unsqueeze(0).expand_as(slot)[m]
    sl = slot[m]
    for c in range(0, sl.numel(), chunk):
        s_, t_ = sl[c:c + chunk], tok[c:c + chunk]
        if fp8:
            assert torch.equal(_canon_e4m3(got[s_]), _canon_e4m3(ref[t_]))
            assert torch.equal(got_sc[s_], ref_sc[t_])
        else:
            assert torch.equal(got[s_], ref[t_])
    if recv_w is not None:
        w_d = torch.from_numpy(w).cuda()
        assert torch.equal(recv_w[sl].view(torch.int32), w_d[tok, kk].view(torch.int32))
    if zero_padding:
        used = int(ora["expert_start"][-1])
        pad = torch.from_numpy(np.nonzero(ora["src_info"][:used, 0] < 0)[0]).cuda().long()
        if pad.numel():
            assert int((got[pad] != 0).sum()) == 0
            if fp8:
                assert int((got_sc[pad] != 0).sum()) == 0
            if recv_w is not None:
                assert int((recv_w[pad] != 0).sum()) == 0


@pytest.mark.parametrize("name", ["sweep16k", "sweep4k", "prefill"])
def test_dispatch_bf16_full_size(ep, name):
    """Every row in use at full size against the oracle's rows."""
    wl = workloads.WORKLOADS[name]
    inp, cfg, L, ora, recv_x, _, recv_w = _dispatch_case(ep, wl, False)
    assert_layout_equal(L, ora, wl.num_tokens)
    assert_rows_equal_oracle(inp, ora, False, recv_x, recv_w=recv_w)


@pytest.mark.parametrize("name,zp", [("decode", False), ("ragged_fp8", True),
                                     ("ragged_fp8", False), ("wide_experts", True),
                                     ("skew_small", False), ("skew", False),
                                     ("sweep1k_fp8", False), ("sweep16k_fp8", False),
                                     ("decode", True)])
def test_dispatch_fp8_bit_exact(ep, name, zp):
    wl = workloads.WORKLOADS.get(name) or MEDIUM[name]
    inp, cfg, L, ora, recv_q, recv_s, recv_w = _dispatch_case(ep, wl, zp)
    assert_rows_equal_oracle(inp, ora, True, recv_q, recv_s, recv_w, zero_padding=zp)
    if wl.num_tokens * wl.num_topk <= 20000:
        # and the oracle's own dispatch call, row for row
        used = int(ora["expert_start"][-1])
        ref_q, ref_s, ref_w = oracle.dispatch_fp8(inp["x"], inp["topk_weights"], ora,
                                                  zero_padding=zp)
        rows = ora["src_info"][:used, 0] >= 0
        if zp:
            rows[:] = True
        assert np.array_equal(recv_q[:used].cpu().numpy()[rows], ref_q[:used][rows])
        assert np.array_equal(recv_s[:used].cpu().numpy()[rows].view(np.uint32),
                              ref_s[:used][rows].view(np.uint32))
        assert np.array_equal(recv_w[:used].cpu().numpy()[rows], ref_w[:used][rows])


def _special_fp8_rows():
    """Zero blocks, saturation-size values, tiny values, signed zeros, rows
    whose block scales lie on both sides of 2^-100 (below it the dispatch
    divides; above it, reciprocal product plus FMA correction), and blocks
    holding +-inf or NaN next to finite values."""
    T, H = 22, 512
    rng = np.random.default_rng(12)
    xf = rng.standard_normal((T, H)).astype(np.float32)
    xf[0] = 0.0                                 # all-zero row: scale 0, q 0
    xf[1, :128] = 0.0                           # one zero block
    xf[2] *= 1e30                               # huge magnitudes
    xf[3] *= 1e-30                              # bf16 subnormal range
    xf[4, ::2] = -0.0
    xf[5, :] = 448.0 * np.sign(xf[5])           # every element at amax
    xf[6, 5] = 3.0e38                           # one block dominated by one value
    for r, e in zip(range(8, 16), [-90, -95, -99, -100, -101, 60, 100, 120]):
        xf[r] *= np.float32(2.0 ** e)
    # non-finite values: the block scale is +inf, finite neighbours encode
    # as +-0, the infinities themselves as NaN codes (inf / inf)
    xf[16, 3] = np.inf                          # +inf in block 0
    xf[16, 130] = -np.inf                       # -inf in block 1
    xf[16, 300] = np.inf                        # both signs in block 2
    xf[16, 301] = -np.inf
    xf[17, :] = np.inf                          # a whole row of +inf
    xf[18, ::3] = -np.inf                       # -inf every third element
    xf[19, 7] = np.nan                          # NaN next to finite values:
    xf[19, 200] = np.nan                        #   ignored by amax
    xf[20, 9] = np.nan                          # NaN and inf in one block
    xf[20, 10] = np.inf
    xf[21, :128] = np.nan                       # an all-NaN block: scale 0
    return workloads.to_bf16_bits(xf)


def test_dispatch_fp8_special_rows(ep):
    x = _special_fp8_rows()
    T, H = x.shape
    idx = np.array([[t % 4, 4 + t % 4] for t in range(T)], np.int64)
    w = np.full((T, 2), 0.5, np.float32)
    wl = workloads.Workload("fp8s", T, H, 8, 2, 2, True, expert_alignment=4)
    cfg = cfg_of(ep, wl, zero_padding=True)
    ora = oracle_layout(wl, idx, cfg.capacity)
    inp = {"x": x, "topk_weights": w}
    ref_q, ref_s, ref_w = oracle.dispatch_fp8(x, w, ora, zero_padding=True)
    used = int(ora["expert_start"][-1])
    # the separate calls, and layout and dispatch in one call (one kernel here)
    L = run_layout(ep, cfg, idx)
    got = [ep.dispatch(cfg, L, dev_bf16(x), dev(w))]
    L2, rq2, rs2, rw2 = ep.layout_and_dispatch(cfg, dev(idx), dev_bf16(x), dev(w))
    torch.cuda.synchronize()
    assert ep.check_error(L2) == ep.EP_OK
    assert_layout_equal(L2, ora, T)
    got.append((rq2, rs2, rw2))
    for rq, rs, rw in got:
        assert_rows_equal_oracle(inp, ora, True, rq, rs, rw, zero_padding=True)
        q = rq[:used].cpu().numpy()
        nan_ref = (ref_q[:used] & 0x7F) == 0x7F
        assert np.array_equal((q & 0x7F) == 0x7F, nan_ref)
        assert np.array_equal(q[~nan_ref], ref_q[:used][~nan_ref])
        assert np.array_equal(rs[:used].cpu().numpy().view(np.uint32),
                              ref_s[:used].view(np.uint32))
        assert np.array_equal(rw[:used].cpu().numpy(), ref_w[:used])
    # the readings themselves: an infinite block has scale +inf and its
    # finite elements encode as +-0
    r16 = ora["slot_of"][16, 0]
    assert np.all(np.isinf(ref_s[r16, :3])) and ref_s[r16, 3] != np.inf
    assert set(np.unique(ref_q[r16, :128][np.arange(128) != 3])) <= {0x00, 0x80}


def test_dispatch_reuses_layout_and_stream(ep):
    wl = MEDIUM["ragged_bf16"]
    inp = inputs(wl)
    cfg = cfg_of(ep, wl, zero_padding=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        L = ep.get_layout(cfg, dev(inp["topk_idx"]))
        x = dev_bf16(inp["x"])
        a, _, _ = ep.dispatch(cfg, L, x, want_weights=False)
        b, _, _ = ep.dispatch(cfg, L, x, want_weights=False)
    s.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# --------------------------------------------------------------------------
# combine
# --------------------------------------------------------------------------

def _expert_out(cfg, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 + seed)
    return torch.randn((cfg.capacity, cfg.hidden), generator=g, device="cuda",
                       dtype=torch.float32).to(torch.bfloat16)


@pytest.mark.parametrize("name,weighted", [
    ("tiny", True), ("tiny", False), ("ragged_bf16", True), ("ragged_fp8", True),
    ("k1_e_eq_r", True), ("wide_experts", True), ("skew_small", False), ("decode", True)])
def test_combine_full_compare(ep, name, weighted):
    wl = workloads.WORKLOADS.get(name) or MEDIUM[name]
    inp = inputs(wl)
    cfg = cfg_of(ep, wl)
    L = run_layout(ep, cfg, inp["topk_idx"])
    Y = _expert_out(cfg, 1)
    w = dev(inp["topk_weights"]) if weighted else None
    y = ep.combine(cfg, L, Y, w)
    torch.cuda.synchronize()
    ora = oracle_layout(wl, inp["topk_idx"], cfg.capacity)
    ref = oracle.combine(host_u16(Y), inp["topk_weights"] if weighted else None, ora["slot_of"])
    got = host_u16(y)
    assert_combine_close(got, ref)
    assert np.array_equal(got, ref)   # expected bit-exact (same fold, same cast)


@pytest.mark.parametrize("name", ["prefill", "skew", "sweep16k", "sweep1k"])
def test_combine_full_size(ep, name):
    """Every token at full size against the oracle's fold."""
    wl = workloads.WORKLOADS[name]
    inp = inputs(wl)
    cfg = cfg_of(ep, wl)
    L = run_layout(ep, cfg, inp["topk_idx"])
    Y = _expert_out(cfg, 2)
    y = ep.combine(cfg, L, Y, dev(inp["topk_weights"]))
    torch.cuda.synchronize()
    ora = oracle_layout(wl, inp["topk_idx"], cfg.capacity)
    used = int(ora["expert_start"][-1])
    ref = oracle.combine(host_u16(Y[:used]), inp["topk_weights"], ora["slot_of"])
    got = host_u16(y)
    assert_combine_close(got, ref)
    assert np.array_equal(got, ref)


def test_combine_non_finite_rows(ep):
    """Expert rows holding +-inf and NaN: the fold propagates them as the
    oracle's does (inf + -inf and 0 * inf give NaN); NaN results compare by
    NaN-ness (the sign of an invalid operation's NaN is not fixed by IEEE),
    everything else bit-exact."""
    wl = MEDIUM["ragged_bf16"]
    inp = inputs(wl)
    cfg = cfg_of(ep, wl)
    L = run_layout(ep, cfg, inp["topk_idx"])
    Yh = host_u16(_expert_out(cfg, 3))
    rng = np.random.default_rng(14)
    cells = rng.integers(0, Yh.size, 4000)
    Yh.reshape(-1)[cells[:1500]] = 0x7F80          # +inf
    Yh.reshape(-1)[cells[1500:3000]] = 0xFF80      # -inf
    Yh.reshape(-1)[cells[3000:]] = 0x7FC0          # NaN
    w = inp["topk_weights"].copy()
    w[::7, 0] = 0.0                                # 0 * inf
    y = ep.combine(cfg, L, dev_bf16(Yh), dev(w))
    torch.cuda.synchronize()
    ora = oracle_layout(wl, inp["topk_idx"], cfg.capacity)
    ref = oracle.combine(Yh, w, ora["slot_of"])
    got = host_u16(y)
    nan = lambda u: ((u & 0x7F80) == 0x7F80) & ((u & 0x7F) != 0)
    assert nan(ref).any() and ((ref & 0x7FFF) == 0x7F80).any()
    assert np.array_equal(nan(got), nan(ref))
    assert np.array_equal(got[~nan(ref)], ref[~nan(ref)])


@pytest.mark.parametrize("name", ["prefill", "sweep16k", "decode"])
def test_identity_experts_round_trip(ep, name):
    """dispatch -> identity experts -> combine returns x bit-exactly when the
    gates sum to 1 (unmasked routing), for every token at full size; for FP8
    dispatch the bf16 round trip is checked on the bf16 path of the same
    routing."""
    wl = workloads.WORKLOADS[name].with_(use_fp8_dispatch=False)
    inp = inputs(wl)
    cfg = cfg_of(ep, wl)
    L = run_layout(ep, cfg, inp["topk_idx"])
    x = dev_bf16(inp["x"])
    w = dev(inp["topk_weights"])
    recv_x, _, _ = ep.dispatch(cfg, L, x, w)
    y = ep.combine(cfg, L, recv_x, w)
    torch.cuda.synchronize()
    # bit-exact, with -0.0 returned as +0.0 (the fold starts from +0.0)
    xi = x.view(torch.int16)
    want = torch.where(xi == -32768, torch.zeros_like(xi), xi)
    assert torch.equal(y.view(torch.int16), want)


# --------------------------------------------------------------------------
# extreme configurations: largest hidden size, one expert, every expert
# selected, largest alignment, one token -- the whole path against the oracle
# --------------------------------------------------------------------------

EXTREME = {
    "h_max_bf16": workloads.Workload("h_max_bf16", 24, 49152, 8, 2, 2, False,
                                     expert_alignment=4),
    "h_max_fp8": workloads.Workload("h_max_fp8", 24, 49152, 8, 2, 2, True,
                                    expert_alignment=4),
    # rows of 2^20 channels (the widest accepted; 2 MB bf16 rows)
    "h_2p20_bf16": workloads.Workload("h_2p20", 6, 1 << 20, 4, 2, 2, False, expert_alignment=2),
    "h_2p20_fp8": workloads.Workload("h_2p20_fp8", 6, 1 << 20, 4, 2, 2, True, expert_alignment=2),
    "one_expert": workloads.Workload("one_expert", 100, 256, 1, 1, 1, False,
                                     expert_alignment=1),
    "k_eq_e": workloads.Workload("k_eq_e", 64, 256, 32, 32, 4, False, expert_alignment=16),
    "align_max": workloads.Workload("align_max", 300, 128, 16, 4, 4, True,
                                    expert_alignment=1024, mask_frac=0.1),
    "one_token_bf16": workloads.Workload("one_token_bf16", 1, 7168, 256, 8, 8, False),
    "one_token_fp8": workloads.Workload("one_token_fp8", 1, 7168, 256, 8, 8, True),
}


@pytest.mark.parametrize("name", list(EXTREME))
@pytest.mark.parametrize("zp", [False, True])
def test_extreme_configs_whole_path(ep, name, zp):
    wl = EXTREME[name]
    inp = workloads.make_inputs(wl, seed=3)
    cfg = cfg_of(ep, wl, zero_padding=zp)
    L = run_layout(ep, cfg, inp["topk_idx"])
    ora = oracle_layout(wl, inp["topk_idx"], cfg.capacity)
    assert_layout_equal(L, ora, wl.num_tokens)
    w = dev(inp["topk_weights"])
    recv, recv_s, recv_w = ep.dispatch(cfg, L, dev_bf16(inp["x"]), w)
    Y = _expert_out(cfg, 2)
    y = ep.combine(cfg, L, Y, w)
    torch.cuda.synchronize()
    used = int(ora["expert_start"][-1])
    rows = np.arange(used) if zp else np.nonzero(ora["src_info"][:used, 0] >= 0)[0]
    if wl.use_fp8_dispatch:
        ref_q, ref_s, ref_w = oracle.dispatch_fp8(inp["x"], inp["topk_weights"], ora,
                                                  zero_padding=zp)
        assert np.array_equal(recv.cpu().numpy()[rows], ref_q[rows])
        assert np.array_equal(recv_s.cpu().numpy()[rows].view(np.uint32),
                              ref_s[rows].view(np.uint32))
    else:
        ref_x, ref_w = oracle.dispatch_bf16(inp["x"], inp["topk_weights"], ora,
                                            zero_padding=zp)
        assert np.array_equal(host_u16(recv)[rows], ref_x[rows])
    assert np.array_equal(recv_w.cpu().numpy()[rows].view(np.uint32),
                          ref_w[rows].view(np.uint32))
    ref_y = oracle.combine(host_u16(Y), inp["topk_weights"], ora["slot_of"])
    assert np.array_equal(host_u16(y), ref_y)


# --------------------------------------------------------------------------
# layout and dispatch in one call: fused for small inputs, the two paths in
# turn for larger ones -- the same layout and rows as separate calls
# --------------------------------------------------------------------------

FUSED = ["tiny", "decode", "ragged_fp8", "small_edge", "k1_e_eq_r", "wide_ranks_small",
         "k_eq_e", "one_token_bf16", "one_token_fp8", "past_small_edge", "prefill"]


@pytest.mark.parametrize("name", FUSED)
@pytest.mark.parametrize("zp", [False, True])
def test_layout_and_dispatch_equals_separate_calls(ep, name, zp):
    wl = workloads.WORKLOADS.get(name) or MEDIUM.get(name) or EXTREME[name]
    inp = inputs(wl)
    cfg = cfg_of(ep, wl, zero_padding=zp)
    idx, x, w = dev(inp["topk_idx"]), dev_bf16(inp["x"]), dev(inp["topk_weights"])
    L1 = ep.get_layout(cfg, idx, sync=True)
    rx1, rs1, rw1 = ep.dispatch(cfg, L1, x, w)
    L2, rx2, rs2, rw2 = ep.layout_and_dispatch(cfg, idx, x, w)
    torch.cuda.synchronize()
    assert ep.check_error(L2) == ep.EP_OK
    ora = oracle_layout(wl, inp["topk_idx"], cfg.capacity)
    assert_layout_equal(L2, ora, wl.num_tokens)
    used = int(ora["expert_start"][-1])
    rows = np.arange(used) if zp else np.nonzero(ora["src_info"][:used, 0] >= 0)[0]
    # against the oracle directly, then against the separate calls
    assert_rows_equal_oracle(inp, ora, cfg.use_fp8_dispatch, rx2, rs2, rw2, zero_padding=zp)
    r = torch.from_numpy(rows).long().cuda()
    assert torch.equal(rx2[r].view(torch.uint8), rx1[r].view(torch.uint8))
    if cfg.use_fp8_dispatch:
        assert torch.equal(rs2[r].view(torch.int32), rs1[r].view(torch.int32))
    assert torch.equal(rw2[r].view(torch.int32), rw1[r].view(torch.int32))

