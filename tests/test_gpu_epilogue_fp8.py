"""GPU parity of the combine epilogue (bias terms, gate-weight return) and
the FP8 dispatch options (column-major scales, pre-quantised input) against
the CPU oracle, bit for bit, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import load_build_module

    load_build_module().build()
    import combine_get_layout_gb300 as ep

    return ep


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(u16):
    return dev(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


CASES = {
    "ragged": workloads.Workload("ragged", 1000, 1024, 64, 8, 8, False,
                                 expert_alignment=16, mask_frac=0.07),
    "decode": workloads.WORKLOADS["decode"].with_(use_fp8_dispatch=False),
    "small_k1": workloads.Workload("small_k1", 37, 256, 16, 1, 4, False, expert_alignment=8),
    "h_2p20": workloads.Workload("h_2p20", 6, 1 << 20, 4, 2, 2, False, expert_alignment=2),
}


def _setup(ep, wl, zero_padding=False, seed=0):
    inp = workloads.make_inputs(wl, seed=seed)
    cfg = ep.Config(wl.num_tokens, wl.hidden, wl.num_topk, wl.num_experts, wl.num_ranks,
                    wl.expert_alignment, wl.use_fp8_dispatch, zero_padding)
    L = ep.get_layout(cfg, dev(inp["topk_idx"]), sync=True)
    ora = oracle.layout(inp["topk_idx"], wl.num_experts, wl.num_ranks,
                        wl.expert_alignment, cap=cfg.capacity)
    assert ora["status"] == oracle.OK
    return inp, cfg, L, ora


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("nbias", [0, 1, 2, -1])
def test_combine_epilogue_bit_exact(ep, name, nbias):
    wl = CASES[name]
    inp, cfg, L, ora = _setup(ep, wl)
    rng = np.random.default_rng(21)
    T, H = wl.num_tokens, wl.hidden
    Yh = workloads.to_bf16_bits(rng.standard_normal((cfg.capacity, H)).astype(np.float32))
    b0 = workloads.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    b1 = workloads.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    x = dev_bf16(inp["x"])
    w = dev(inp["topk_weights"])
    _, _, recv_w = ep.dispatch(cfg, L, x, w)
    # nbias -1: only the second bias given
    use0 = b0 if nbias in (1, 2) else None
    use1 = b1 if nbias in (2, -1) else None
    y, cw = ep.combine_epilogue(cfg, L, dev_bf16(Yh), w,
                                bias0=None if use0 is None else dev_bf16(use0),
                                bias1=None if use1 is None else dev_bf16(use1),
                                recv_w=recv_w, want_weights=True)
    torch.cuda.synchronize()
    _, ref_rw = oracle.dispatch_bf16(inp["x"], inp["topk_weights"], ora)
    ref_y, ref_cw = oracle.combine_epilogue(Yh, inp["topk_weights"], ora["slot_of"],
                                            bias0=use0, bias1=use1, recv_w=ref_rw)
    assert np.array_equal(host_u16(y), ref_y)
    assert np.array_equal(cw.cpu().numpy(), ref_cw)
    if nbias == 0:
        plain = ep.combine(cfg, L, dev_bf16(Yh), w)
        assert torch.equal(plain.view(torch.int16), y.view(torch.int16))


FP8 = {
    "ragged_fp8": workloads.Workload("ragged_fp8", 333, 1024, 32, 4, 4, True,
                                     expert_alignment=8, mask_frac=0.1),
    "decode": workloads.WORKLOADS["decode"],
    "odd_cap": workloads.Workload("odd_cap", 5, 256, 6, 3, 3, True, expert_alignment=3),
    "h_2p20_fp8": workloads.Workload("h_2p20_fp8", 6, 1 << 20, 4, 2, 2, True, expert_alignment=2),
}


@pytest.mark.parametrize("name", list(FP8))
@pytest.mark.parametrize("zp", [False, True])
def test_fp8_col_major_scales(ep, name, zp):
    wl = FP8[name]
    inp, cfg, L, ora = _setup(ep, wl, zero_padding=zp)
    x = dev_bf16(inp["x"])
    w = dev(inp["topk_weights"])
    q_r, s_r, w_r = ep.dispatch_fp8(cfg, L, x=x, topk_weights=w)
    q_c, s_c, w_c = ep.dispatch_fp8(cfg, L, x=x, topk_weights=w, scale_col_major=True)
    torch.cuda.synchronize()
    ld = ep.ep_scale_ld(cfg.c())
    assert ld == oracle.scale_ld(cfg.capacity) and tuple(s_c.shape) == (wl.hidden // 128, ld)
    ref_q, ref_s, ref_w = oracle.dispatch_fp8(inp["x"], inp["topk_weights"], ora, zero_padding=zp)
    used = int(ora["expert_start"][-1])
    rows = np.ones(used, bool) if zp else ora["src_info"][:used, 0] >= 0
    # row-major through the new entry point: the fused definition
    assert np.array_equal(q_r.cpu().numpy()[:used][rows], ref_q[:used][rows])
    assert np.array_equal(s_r.cpu().numpy()[:used][rows].view(np.uint32),
                          ref_s[:used][rows].view(np.uint32))
    # column-major: the oracle's transpose of the same scales
    col = oracle.scales_to_col_major(ref_s)
    got = s_c.cpu().numpy()
    assert np.array_equal(got[:, :used][:, rows].view(np.uint32),
                          col[:, :used][:, rows].view(np.uint32))
    assert np.array_equal(q_c.cpu().numpy()[:used][rows], ref_q[:used][rows])
    assert np.array_equal(w_c.cpu().numpy()[:used][rows], ref_w[:used][rows])


@pytest.mark.parametrize("name", list(FP8))
@pytest.mark.parametrize("col", [False, True])
def test_fp8_prequantised_input(ep, name, col):
    wl = FP8[name]
    inp, cfg, L, ora = _setup(ep, wl, zero_padding=True)
    rng = np.random.default_rng(31)
    T, H = wl.num_tokens, wl.hidden
    x_q = rng.integers(0, 256, (T, H), dtype=np.uint8)
    x_q[(x_q & 0x7F) == 0x7F] = 0x42           # no NaN codes needed for a bit copy
    x_s = rng.random((T, H // 128)).astype(np.float32)
    w = dev(inp["topk_weights"])
    q, s, rw = ep.dispatch_fp8(cfg, L, x_q=dev(x_q), x_scale=dev(x_s), topk_weights=w,
                               scale_col_major=col)
    torch.cuda.synchronize()
    ref_q, ref_s, ref_w = oracle.dispatch_fp8_prequant(x_q, x_s, inp["topk_weights"], ora,
                                                       zero_padding=True)
    used = int(ora["expert_start"][-1])
    assert np.array_equal(q.cpu().numpy()[:used], ref_q[:used])
    got_s = s.cpu().numpy()
    want_s = oracle.scales_to_col_major(ref_s)[:, :used] if col else ref_s[:used]
    got_s = got_s[:, :used] if col else got_s[:used]
    assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32))
    assert np.array_equal(rw.cpu().numpy()[:used], ref_w[:used])


def test_fp8_dispatch_argument_checks(ep):
    wl = FP8["ragged_fp8"]
    inp, cfg, L, ora = _setup(ep, wl)
    x = dev_bf16(inp["x"])
    xq = torch.zeros((wl.num_tokens, wl.hidden), dtype=torch.uint8, device="cuda")
    with pytest.raises(ep.EpError):      # both input forms
        ep.dispatch_fp8(cfg, L, x=x, x_q=xq, x_scale=torch.zeros(
            (wl.num_tokens, wl.hidden // 128), device="cuda"))
    with pytest.raises(ep.EpError):      # scales missing
        ep.dispatch_fp8(cfg, L, x_q=xq)


def test_fp8_quotient_exhaustive(ep):
    """The dispatch's x / scale (reciprocal product plus one FMA correction
    where the scale allows it, IEEE division where it does not) gives the
    E4M3 code of the IEEE division for every positive bf16 block maximum,
    finite or +inf, and every bf16 value in its block (about 2^31 pairs: the
    whole non-NaN input domain, so the FP8 payloads equal the oracle's codes
    for every input without NaN; NaN elements give NaN codes on both sides).
    The fp32 quotients themselves may differ in the last bit; those counts
    are reported, not asserted."""
    counts = torch.zeros(4, dtype=torch.int64, device="cuda")
    first = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = ep.ep_selftest_fp8_quotient(counts.data_ptr(), first.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == ep.EP_OK
    torch.cuda.synchronize()
    c = counts.cpu().numpy()
    f = int(first.item())
    assert c[0] == 0, (c, hex(f & 0xFFFFFFFF))
    print(f"fp32 quotients differing (same E4M3 codes): {int(c[1])}, "
          f"of which with a normal IEEE quotient: {int(c[2])}")

