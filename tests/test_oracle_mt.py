"""The multi-threaded driver of the oracle (the timed CPU baseline's
multi-core leg) gives the single-threaded oracle's results bit for bit: it
only runs the same functions on disjoint token slices."""

import numpy as np
import pytest

import oracle
import workloads

CASES = {
    "ragged": workloads.Workload("ragged", 601, 256, 32, 4, 8, False, expert_alignment=8,
                                 mask_frac=0.07),
    "fp8": workloads.Workload("fp8", 333, 512, 16, 3, 4, True, expert_alignment=4,
                              mask_frac=0.1),
    "few_tokens": workloads.Workload("few_tokens", 3, 128, 8, 2, 2, False, expert_alignment=4),
}


def _setup(wl):
    inp = workloads.make_inputs(wl, seed=5)
    cap = oracle.recv_capacity(wl.num_tokens, wl.num_topk, wl.num_experts,
                               wl.expert_alignment)
    lay = oracle.layout(inp["topk_idx"], wl.num_experts, wl.num_ranks, wl.expert_alignment,
                        cap=cap)
    assert lay["status"] == oracle.OK
    return inp, lay


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("nthreads", [2, 5, 16])
@pytest.mark.parametrize("zp", [False, True])
def test_dispatch_mt_equals_single(name, nthreads, zp):
    wl = CASES[name]
    inp, lay = _setup(wl)
    if wl.use_fp8_dispatch:
        a = oracle.dispatch_fp8(inp["x"], inp["topk_weights"], lay, zero_padding=zp)
        b = oracle.dispatch_fp8(inp["x"], inp["topk_weights"], lay, zero_padding=zp,
                                nthreads=nthreads)
    else:
        a = oracle.dispatch_bf16(inp["x"], inp["topk_weights"], lay, zero_padding=zp)
        b = oracle.dispatch_bf16(inp["x"], inp["topk_weights"], lay, zero_padding=zp,
                                 nthreads=nthreads)
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.uint8), v.view(np.uint8))


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("nthreads", [2, 7])
@pytest.mark.parametrize("weighted", [True, False])
def test_combine_mt_equals_single(name, nthreads, weighted):
    wl = CASES[name]
    inp, lay = _setup(wl)
    rng = np.random.default_rng(8)
    Y = workloads.to_bf16_bits(rng.standard_normal((lay["cap"], wl.hidden)))
    w = inp["topk_weights"] if weighted else None
    a = oracle.combine(Y, w, lay["slot_of"])
    b = oracle.combine(Y, w, lay["slot_of"], nthreads=nthreads)
    assert np.array_equal(a, b)
