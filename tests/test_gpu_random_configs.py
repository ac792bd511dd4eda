"""GPU parity over seeded random configurations: token counts on both sides
of the one-launch layout's limit, expert and rank counts, top-k, expert
alignments, row widths, masking, zero padding, bf16 and FP8 rows.  Each case
runs the whole path through the C ABI -- layout, dispatch (separate calls
and the one-call layout + dispatch), combine -- and compares every output
element with the oracle on the same inputs."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import (assert_layout_equal, assert_rows_equal_oracle, cfg_of, dev,
                             dev_bf16, host_u16, oracle_layout)

pytestmark = pytest.mark.gpu

N_CASES = 40


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import load_build_module

    load_build_module().build()
    import combine_get_layout_gb300 as ep

    return ep


def random_case(i):
    """Configuration i of the sweep (seeded, so every run draws the same)."""
    rng = np.random.default_rng(1000 + i)
    R = int(rng.choice([1, 2, 3, 4, 8, 16, 32, 64]))
    E = R * int(rng.choice([1, 2, 3, 4, 8, 16]))
    K = int(rng.integers(1, min(E, 32) + 1))
    fp8 = bool(rng.integers(0, 2))
    H = 128 * int(rng.integers(1, 9)) if fp8 else 8 * int(rng.integers(1, 129))
    # about half the cases on each side of 4096 (t, k) pairs
    T = int(rng.integers(1, 4096 // K + 1)) if i % 2 == 0 else int(rng.integers(4096 // K + 1, 3 * 4096 // K + 2))
    A = int(rng.choice([1, 2, 4, 16, 128, 256]))
    mask = float(rng.choice([0.0, 0.05, 0.5]))
    zp = bool(rng.integers(0, 2))
    wl = workloads.Workload(f"rand{i}", T, H, E, K, R, fp8, expert_alignment=A, mask_frac=mask)
    idx = workloads.random_routes(rng, T, E, K, mask)
    x = workloads.to_bf16_bits(rng.standard_normal((T, H)) * float(rng.choice([1.0, 1e-3, 1e3])))
    w = rng.random((T, K)).astype(np.float32)
    return wl, zp, {"topk_idx": idx, "x": x, "topk_weights": w}


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_config_whole_path(ep, i):
    wl, zp, inp = random_case(i)
    cfg = cfg_of(ep, wl, zero_padding=zp)
    ora = oracle_layout(wl, inp["topk_idx"], cfg.capacity)
    idx, x, w = dev(inp["topk_idx"]), dev_bf16(inp["x"]), dev(inp["topk_weights"])
    L = ep.get_layout(cfg, idx, sync=True)
    assert_layout_equal(L, ora, wl.num_tokens)
    rx, rs, rw = ep.dispatch(cfg, L, x, w)
    L2, rx2, rs2, rw2 = ep.layout_and_dispatch(cfg, idx, x, w)
    torch.cuda.synchronize()
    assert ep.check_error(L2) == ep.EP_OK
    assert_layout_equal(L2, ora, wl.num_tokens)
    for q, s, ww in ((rx, rs, rw), (rx2, rs2, rw2)):
        assert_rows_equal_oracle(inp, ora, wl.use_fp8_dispatch, q, s, ww, zero_padding=zp)
    # combine of seeded expert rows, weighted
    g = torch.Generator(device="cuda")
    g.manual_seed(77 + i)
    Y = torch.randn((cfg.capacity, wl.hidden), generator=g, device="cuda").to(torch.bfloat16)
    y = ep.combine(cfg, L, Y, w)
    torch.cuda.synchronize()
    used = int(ora["expert_start"][-1])
    ref = oracle.combine(host_u16(Y[:max(used, 1)]), inp["topk_weights"], ora["slot_of"])
    assert np.array_equal(host_u16(y), ref)


def test_random_cases_cover_both_layout_paths():
    sizes = [random_case(i)[0] for i in range(N_CASES)]
    small = sum(wl.num_tokens * wl.num_topk <= 4096 for wl in sizes)
    assert 0 < small < N_CASES
    assert any(wl.use_fp8_dispatch for wl in sizes) and not all(wl.use_fp8_dispatch for wl in sizes)
