"""GPU parity of the backward pair (ep_dispatch_backward, ep_combine_backward)
against the CPU oracle.

Bars: grad_x and the grad_expert_out rows are bit-exact (same fp32 fold, same
products, same single bf16 rounding); gate gradients are fp32 dot products
over H whose summation order differs from the oracle's double-precision sum,
so they are held to the fp32 summation error bound
|err| <= (H + 2) * 2^-24 * sum_i |dy_i * Y_i|, and must be identical from run
to run (fixed reduction order)."""

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


def bits(a, rng):
    return workloads.to_bf16_bits(rng.standard_normal(a).astype(np.float32))


CASES = {
    "ragged": workloads.Workload("ragged", 1000, 1024, 64, 8, 8, False,
                                 expert_alignment=16, mask_frac=0.07),
    "k12": workloads.Workload("k12", 300, 512, 48, 12, 6, False, expert_alignment=8,
                              mask_frac=0.1),
    "decode": workloads.WORKLOADS["decode"].with_(use_fp8_dispatch=False),
    "k1": workloads.Workload("k1", 257, 256, 16, 1, 16, False, expert_alignment=1),
    "k_eq_e": workloads.Workload("k_eq_e", 64, 256, 32, 32, 4, False, expert_alignment=16),
    "prefill": workloads.WORKLOADS["prefill"],
    "h_2p20": workloads.Workload("h_2p20", 6, 1 << 20, 4, 2, 2, False, expert_alignment=2),
}


def _setup(ep, wl, zp=False):
    inp = workloads.make_inputs(wl, seed=0)
    cfg = ep.Config(wl.num_tokens, wl.hidden, wl.num_topk, wl.num_experts, wl.num_ranks,
                    wl.expert_alignment, False, zp)
    L = ep.get_layout(cfg, dev(inp["topk_idx"]), sync=True)
    ora = oracle.layout(inp["topk_idx"], wl.num_experts, wl.num_ranks,
                        wl.expert_alignment, cap=cfg.capacity)
    assert ora["status"] == oracle.OK
    return inp, cfg, L, ora


def _tokens(wl):
    if wl.num_tokens <= 1000:
        return np.arange(wl.num_tokens)
    rng = np.random.default_rng(5)
    return np.unique(np.concatenate([[0, wl.num_tokens - 1], rng.choice(wl.num_tokens, 256)]))


@pytest.mark.parametrize("name", ["ragged", "k12", "decode", "k1", "k_eq_e", "h_2p20"])
def test_dispatch_backward_bit_exact(ep, name):
    wl = CASES[name]
    inp, cfg, L, ora = _setup(ep, wl)
    rng = np.random.default_rng(41)
    G = bits((cfg.capacity, wl.hidden), rng)
    Gw = rng.standard_normal(cfg.capacity).astype(np.float32)
    gx, gw = ep.dispatch_backward(cfg, L, dev_bf16(G), dev(Gw))
    torch.cuda.synchronize()
    ref_x, ref_w = oracle.dispatch_backward(G, ora["slot_of"], Gw)
    assert np.array_equal(host_u16(gx), ref_x)
    assert np.array_equal(gw.cpu().numpy(), ref_w)


def _check_grad_w(got, dy, Y, so, tokens, H):
    for i, t in enumerate(tokens):
        for k in range(so.shape[1]):
            s = so[t, k]
            if s < 0:
                assert got[i, k] == 0
                continue
            a = oracle.bf16_to_f32_array(dy[t]).astype(np.float64)
            b = oracle.bf16_to_f32_array(Y[s]).astype(np.float64)
            exact = float((a * b).sum())
            bound = (H + 2) * 2.0**-24 * float(np.abs(a * b).sum()) + 1e-30
            assert abs(float(got[i, k]) - exact) <= bound, (t, k, got[i, k], exact)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("weighted", [True, False])
def test_combine_backward(ep, name, weighted):
    wl = CASES[name]
    inp, cfg, L, ora = _setup(ep, wl, zp=True)
    T, H = wl.num_tokens, wl.hidden
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    Y = torch.randn((cfg.capacity, H), generator=g, device="cuda").to(torch.bfloat16)
    dy = torch.randn((T, H), generator=g, device="cuda").to(torch.bfloat16)
    w = dev(inp["topk_weights"]) if weighted else None
    gY, gw = ep.combine_backward(cfg, L, dy, w, expert_out=Y)
    gY2, gw2 = ep.combine_backward(cfg, L, dy, w, expert_out=Y)
    torch.cuda.synchronize()
    assert torch.equal(gw.view(torch.int32), gw2.view(torch.int32))   # deterministic
    toks = _tokens(wl)
    so = ora["slot_of"]
    dy_h = host_u16(dy)
    rows = np.unique(so[toks][so[toks] >= 0])
    Y_h = np.zeros((cfg.capacity, H), np.uint16)
    Y_h[rows] = host_u16(Y[torch.from_numpy(rows).long().cuda()])
    sub_so = np.full_like(so, -1)
    sub_so[toks] = so[toks]
    ref_gY, _ = oracle.combine_backward(dy_h, inp["topk_weights"] if weighted else None,
                                        sub_so, cfg.capacity, want_grad_w=False)
    got_gY = host_u16(gY)
    assert np.array_equal(got_gY[rows], ref_gY[rows])
    _check_grad_w(gw.cpu().numpy()[toks], dy_h, Y_h, so, toks, H)
    # alignment gap rows are zero (zero padding is on)
    es, ee = ora["expert_start"], ora["expert_end"]
    for e in range(0, wl.num_experts, max(1, wl.num_experts // 16)):
        assert np.all(got_gY[ee[e]:es[e + 1]] == 0)


def test_unweighted_combine_backward_is_dispatch(ep):
    wl = CASES["ragged"]
    inp, cfg, L, ora = _setup(ep, wl)
    dy = dev_bf16(inp["x"])
    gY, _ = ep.combine_backward(cfg, L, dy, None, want_grad_w=False)
    recv, _, _ = ep.dispatch(cfg, L, dy)
    torch.cuda.synchronize()
    used = int(ora["expert_start"][-1])
    rows = np.nonzero(ora["src_info"][:used, 0] >= 0)[0]
    r = torch.from_numpy(rows).long().cuda()
    assert torch.equal(gY[r].view(torch.int16), recv[r].view(torch.int16))
