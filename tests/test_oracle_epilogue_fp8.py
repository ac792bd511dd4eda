"""Pins for the oracle's combine epilogue (bias terms, gate-weight return) and
FP8 variants (column-major scale layout, pre-quantised input).

Sources: "Deep Dive - DeepEP", "Combine: reverse routing plus reduction"
(zero, one or two bf16 biases in the combine epilogue; optional return of
top-k weights; one final bf16 cast -- the 256 + 1 - 256 case) and
"Precision: FP8 on the wire, BF16 for the reduction" (input as FP8 values
plus scale factors; a column-major scale layout for TMA paths).
"""

import numpy as np

import oracle
import workloads
from workloads import to_bf16_bits


def bf(a):
    return to_bf16_bits(np.asarray(a, np.float32))


def f32(h):
    return oracle.bf16_to_f32_array(h)


def lay_of(idx, E, R, A):
    lay = oracle.layout(np.asarray(idx, np.int64), E, R, A)
    assert lay["status"] == oracle.OK
    return lay


def _case(seed=0, T=24, H=16, E=8, K=3, mask=0.2):
    rng = np.random.default_rng(seed)
    idx = workloads.random_routes(rng, T, E, K, mask_frac=mask)
    lay = lay_of(idx, E, 4, 4)
    Y = bf(rng.standard_normal((lay["cap"], H)))
    w = rng.random((T, K)).astype(np.float32)
    return rng, idx, lay, Y, w


def test_epilogue_without_extras_is_combine():
    rng, idx, lay, Y, w = _case()
    y, cw = oracle.combine_epilogue(Y, w, lay["slot_of"])
    assert np.array_equal(y, oracle.combine(Y, w, lay["slot_of"])) and cw is None


def test_bias_added_in_fp32_after_the_fold(golden):
    # the page's cancellation numbers: a fold of 256, then +1 and -256 as
    # the two biases; one final cast gives 1 (a bf16 subtotal would give 0)
    g = dict(golden("worked_values.txt"))
    a, b, c = [float(v) for v in g["p9_terms"]]
    Y = bf([[a]])
    so = np.array([[0]], np.int32)
    y, _ = oracle.combine_epilogue(Y, None, so, bias0=bf([[b]]), bias1=bf([[c]]))
    assert f32(y)[0, 0] == float(g["p9_single_stage"][0])


def test_bias_closed_forms():
    Y = bf([[1.5, 2.0]])
    so = np.array([[0]], np.int32)
    y, _ = oracle.combine_epilogue(Y, np.array([[1.0]], np.float32), so,
                                   bias0=bf([[0.25, -2.0]]), bias1=bf([[-0.125, 0.0]]))
    assert list(f32(y)[0]) == [1.625, 0.0]
    # all selections masked: the output is the bias itself (exact in bf16)
    so = np.array([[-1, -1]], np.int32)
    b = bf([[3.0, -7.5]])
    y, _ = oracle.combine_epilogue(Y, np.ones((1, 2), np.float32), so, bias0=b)
    assert np.array_equal(y, b)


def test_one_bias_equals_two_with_zero():
    rng, idx, lay, Y, w = _case(1)
    T, H = idx.shape[0], Y.shape[1]
    b = bf(rng.standard_normal((T, H)))
    z = np.zeros((T, H), np.uint16)
    y1, _ = oracle.combine_epilogue(Y, w, lay["slot_of"], bias0=b)
    y2, _ = oracle.combine_epilogue(Y, w, lay["slot_of"], bias0=b, bias1=z)
    assert np.array_equal(y1, y2)


def test_combined_weights_round_trip():
    rng, idx, lay, Y, w = _case(2)
    x = bf(rng.standard_normal((idx.shape[0], Y.shape[1])))
    _, recv_w = oracle.dispatch_bf16(x, w, lay)
    _, cw = oracle.combine_epilogue(Y, w, lay["slot_of"], recv_w=recv_w)
    assert np.array_equal(cw[idx >= 0], w[idx >= 0])
    assert np.all(cw[idx < 0] == 0)


def test_col_major_scales_are_the_transpose():
    rng = np.random.default_rng(3)
    for cap in (1, 3, 4, 5, 1048):
        assert oracle.scale_ld(cap) % 4 == 0
        assert cap <= oracle.scale_ld(cap) < cap + 4
        rm = rng.random((cap, 7)).astype(np.float32)
        col = oracle.scales_to_col_major(rm)
        assert np.array_equal(col[:, :cap], rm.T)


def test_prequant_dispatch_matches_fused_quantisation():
    """Quantising each token once (a one-row-per-token layout) and then
    dispatching the FP8 rows with their scales gives exactly the fused FP8
    dispatch: the two definitions agree."""
    rng = np.random.default_rng(4)
    T, H, E, K = 20, 384, 8, 3
    idx = workloads.random_routes(rng, T, E, K, mask_frac=0.1)
    lay = lay_of(idx, E, 2, 4)
    x = bf(rng.standard_normal((T, H)) * 3)
    one = {"slot_of": np.arange(T, dtype=np.int32).reshape(T, 1), "cap": T,
           "expert_count": np.array([T], np.int32),
           "expert_start": np.array([0, T], np.int32), "expert_end": np.array([T], np.int32)}
    xq, xs, _ = oracle.dispatch_fp8(x, None, one)
    w = rng.random((T, K)).astype(np.float32)
    for zp in (False, True):
        a = oracle.dispatch_fp8(x, w, lay, zero_padding=zp)
        b = oracle.dispatch_fp8_prequant(xq, xs, w, lay, zero_padding=zp)
        used = lay["expert_start"][-1]
        rows = lay["src_info"][:used, 0] >= 0
        if zp:
            rows[:] = True
        for u, v in zip(a, b):
            assert np.array_equal(u[:used][rows].view(np.uint8), v[:used][rows].view(np.uint8))


def test_bias_order_fold_then_b0_then_b1():
    """(fold + b0) + b1, each in fp32: with a fold of 1 + 2^-8 and two biases
    of 2^-24, each add is an fp32 tie that stays at 1 + 2^-8, and the final
    bf16 tie goes to even (1.0).  Adding the biases first (2^-23), or before
    the fold, lands above the bf16 midpoint (1 + 2^-7)."""
    Y = bf([[1.0]])
    w = np.array([[1.0 + 2.0**-8]], np.float32)
    tiny = bf([[2.0**-24]])
    so = np.array([[0]], np.int32)
    y, _ = oracle.combine_epilogue(Y, w, so, bias0=tiny, bias1=tiny)
    assert y[0, 0] == 0x3F80
    # the alternative order, computed here in numpy fp32, differs
    alt = np.float32(np.float32(2.0**-24) + np.float32(2.0**-24)) + np.float32(1.0 + 2.0**-8)
    assert oracle.f32_to_bf16(alt) == 0x3F81
