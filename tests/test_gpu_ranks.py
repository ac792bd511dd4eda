"""GPU parity of the non-expanded (destination-major) stage against the CPU
oracle, bit for bit: rank rows from the layout, dispatch to ranks with the
per-row top-k metadata, expansion to expert rows, the per-rank reduction and
the token-major sum over ranks."""

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
    "tiny": workloads.WORKLOADS["tiny"],
    "ragged": workloads.Workload("ragged", 1000, 1024, 64, 8, 8, False,
                                 expert_alignment=16, mask_frac=0.07),
    "r64": workloads.Workload("r64", 700, 512, 256, 8, 64, False),
    "r64_small": workloads.Workload("r64_small", 300, 512, 256, 8, 64, False,
                                    expert_alignment=8, mask_frac=0.05),
    "prefill": workloads.WORKLOADS["prefill"],
    "skew": workloads.WORKLOADS["skew"].with_(use_fp8_dispatch=False),
    "many_tiles": workloads.Workload("many_tiles", 70000, 8, 256, 8, 8, False),
    # one rank owns every expert; one expert per rank
    "one_rank": workloads.Workload("one_rank", 300, 256, 16, 4, 1, False, expert_alignment=4,
                                   mask_frac=0.05),
    "rank_per_expert": workloads.Workload("rank_per_expert", 200, 256, 16, 4, 16, False,
                                          expert_alignment=4),
    "h_2p20": workloads.Workload("h_2p20", 6, 1 << 20, 4, 2, 2, False, expert_alignment=2),
}


def _setup(ep, wl, noalloc=False, zp=False):
    inp = workloads.make_inputs(wl, seed=0)
    cfg = ep.Config(wl.num_tokens, wl.hidden, wl.num_topk, wl.num_experts, wl.num_ranks,
                    wl.expert_alignment, False, zp)
    L = ep.Layout(cfg, with_ranks=True)
    idx = dev(inp["topk_idx"])
    if noalloc:
        L.c.workspace = None
        st = ep.ep_get_layout_noalloc(cfg.c(), wl.num_tokens, idx.data_ptr(), L.c, None,
                                      torch.cuda.current_stream().cuda_stream)
        assert st == ep.EP_OK
        L.h_expert_count = None
    else:
        ep.get_layout(cfg, idx, layout=L, sync=True)
    torch.cuda.synchronize()
    ora = oracle.layout(inp["topk_idx"], wl.num_experts, wl.num_ranks,
                        wl.expert_alignment, cap=cfg.capacity)
    assert ora["status"] == oracle.OK
    rl = oracle.rank_layout(ora)
    return inp, cfg, L, idx, ora, rl


@pytest.mark.parametrize("name", list(CASES))
def test_rank_rows_bit_exact(ep, name):
    wl = CASES[name]
    inp, cfg, L, idx, ora, rl = _setup(ep, wl)
    assert np.array_equal(L.rank_row_start.cpu().numpy(), rl["rank_row_start"])
    assert np.array_equal(L.rank_slot_of.cpu().numpy()[: wl.num_tokens], rl["rank_slot_of"])
    n = rl["rows"]
    assert np.array_equal(L.rank_src.cpu().numpy()[:n], rl["rank_src"][:n])
    assert n <= ep.ep_rank_rows_capacity(cfg.c())
    # the rest of the layout is unchanged by the rank rows
    assert np.array_equal(L.slot_of.cpu().numpy()[: wl.num_tokens], ora["slot_of"])
    assert np.array_equal(L.tokens_per_rank.cpu().numpy(), ora["tokens_per_rank"])


def test_rank_rows_through_noalloc_entry_point(ep):
    wl = CASES["ragged"]
    inp, cfg, L, idx, ora, rl = _setup(ep, wl, noalloc=True)
    assert np.array_equal(L.rank_slot_of.cpu().numpy()[: wl.num_tokens], rl["rank_slot_of"])
    assert np.array_equal(L.rank_src.cpu().numpy()[: rl["rows"]], rl["rank_src"][: rl["rows"]])


@pytest.mark.parametrize("name", ["tiny", "ragged", "r64", "r64_small", "skew", "one_rank", "h_2p20",
                                  "rank_per_expert"])
def test_dispatch_ranks_and_expand(ep, name):
    wl = CASES[name]
    inp, cfg, L, idx, ora, rl = _setup(ep, wl, zp=True)
    x = dev_bf16(inp["x"])
    w = dev(inp["topk_weights"])
    rank_x, ridx, rw = ep.dispatch_ranks(cfg, L, x, idx, w)
    recv, recv_w = ep.expand(cfg, L, idx, rank_x, rw)
    direct, _, direct_w = ep.dispatch(cfg, L, x, w)
    torch.cuda.synchronize()
    n = rl["rows"]
    ref_x, ref_idx, ref_w = oracle.dispatch_ranks(inp["x"], inp["topk_idx"],
                                                  inp["topk_weights"], rl, wl.num_experts)
    assert np.array_equal(host_u16(rank_x)[:n], ref_x[:n])
    assert np.array_equal(ridx.cpu().numpy()[:n], ref_idx[:n])
    assert np.array_equal(rw.cpu().numpy()[:n], ref_w[:n])
    ref_e, ref_ew = oracle.expand(inp["topk_idx"], ora, rl, ref_x, ref_w, wl.num_experts)
    used = int(ora["expert_start"][-1])
    rows = ora["src_info"][:used, 0] >= 0
    got = host_u16(recv)[:used]
    assert np.array_equal(got[rows], ref_e[:used][rows])
    assert np.all(got[~rows] == 0)                       # zero padding
    assert np.array_equal(recv_w.cpu().numpy()[:used][rows], ref_ew[:used][rows])
    # expand(dispatch_ranks(x)) is the expanded dispatch
    assert torch.equal(recv[:used].view(torch.int16), direct[:used].view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "ragged", "r64", "r64_small", "skew", "prefill", "h_2p20",
                                  "one_rank", "rank_per_expert"])
@pytest.mark.parametrize("weighted", [True, False])
def test_reduce_and_combine_ranks(ep, name, weighted):
    wl = CASES[name]
    inp, cfg, L, idx, ora, rl = _setup(ep, wl)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    Y = torch.randn((cfg.capacity, wl.hidden), generator=g, device="cuda").to(torch.bfloat16)
    w = dev(inp["topk_weights"]) if weighted else None
    rank_y = ep.reduce_ranks(cfg, L, idx, Y, w)
    y = ep.combine_ranks(cfg, L, rank_y)
    torch.cuda.synchronize()
    T = wl.num_tokens
    if T <= 1000:
        toks = np.arange(T)
    else:
        toks = np.unique(np.concatenate([[0, T - 1],
                                         np.random.default_rng(3).choice(T, 200)]))
    so = ora["slot_of"]
    rows = np.unique(so[toks][so[toks] >= 0])
    Yh = np.zeros((cfg.capacity, wl.hidden), np.uint16)
    Yh[rows] = host_u16(Y[torch.from_numpy(rows).long().cuda()])
    # restrict the oracle to the sampled tokens (other tokens' rows unused)
    keep = np.zeros(T, bool)
    keep[toks] = True
    sub_idx = np.where(keep[:, None], inp["topk_idx"], -1)
    sub_rl = dict(rl)
    sub_rl["rank_slot_of"] = np.where(keep[:, None], rl["rank_slot_of"], -1)
    ref_ry = oracle.reduce_ranks(sub_idx, ora, sub_rl, Yh,
                                 inp["topk_weights"] if weighted else None, wl.num_experts)
    rrows = sub_rl["rank_slot_of"][toks]
    rrows = rrows[rrows >= 0]
    got_ry = host_u16(rank_y)
    assert np.array_equal(got_ry[rrows], ref_ry[rrows])
    ref_y = oracle.combine_ranks(sub_rl, ref_ry)
    assert np.array_equal(host_u16(y)[toks], ref_y[toks])


def test_two_stage_cancellation_on_gpu(ep):
    """The pages' 256 + 1 - 256: two experts of rank 0 give 256 and 1, one of
    rank 1 gives -256.  The rank partial rounds to 256 and the two-stage
    result is 0; the single-stage combine gives 1."""
    cfg = ep.Config(1, 8, 3, 4, 2, 1)
    idx = dev(np.array([[0, 1, 2]], np.int64))
    L = ep.get_layout(cfg, idx, sync=True, with_ranks=True)
    so = L.slot_of.cpu().numpy()[0]
    Yh = np.zeros((cfg.capacity, 8), np.float32)
    Yh[so[0]], Yh[so[1]], Yh[so[2]] = 256.0, 1.0, -256.0
    Y = dev_bf16(workloads.to_bf16_bits(Yh))
    rank_y = ep.reduce_ranks(cfg, L, idx, Y, None)
    two = ep.combine_ranks(cfg, L, rank_y)
    one = ep.combine(cfg, L, Y, None)
    torch.cuda.synchronize()
    assert float(rank_y[L.rank_slot_of[0, 0]].float()[0]) == 256.0
    assert float(two.float()[0, 0]) == 0.0
    assert float(one.float()[0, 0]) == 1.0
