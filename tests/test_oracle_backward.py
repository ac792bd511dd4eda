"""Pins for the oracle's backward pair.

Source: "Deep Dive - DeepEP", combine section ("Backward duality provides a
compact consistency check": for the unweighted route operators dispatch and
combine are transposes -- copying rows forward becomes summing their
gradients backward -- and the gate multiplication needs its own gradient).
Pinned by the adjoint identities in both directions, by the statement that
the unweighted combine's transpose is a dispatch, by the 1.90 example of
"Combine: reverse routing plus reduction", and by closed forms.
"""

import numpy as np

import oracle
import workloads
from workloads import to_bf16_bits


def bf(a):
    return to_bf16_bits(np.asarray(a, np.float32))


def f64(h):
    return oracle.bf16_to_f32_array(h).astype(np.float64)


def _case(seed, T=30, H=24, E=8, K=3, mask=0.2):
    rng = np.random.default_rng(seed)
    idx = workloads.random_routes(rng, T, E, K, mask_frac=mask)
    lay = oracle.layout(idx, E, 4, 4)
    assert lay["status"] == oracle.OK
    return rng, idx, lay


def test_dispatch_backward_is_the_transpose():
    rng, idx, lay = _case(0)
    T, H = idx.shape[0], 24
    x = bf(rng.standard_normal((T, H)))
    G = bf(rng.standard_normal((lay["cap"], H)))
    recv_x, _ = oracle.dispatch_bf16(x, None, lay, zero_padding=True)
    gx, _ = oracle.dispatch_backward(G, lay["slot_of"])
    used = lay["expert_start"][-1]
    rows = lay["src_info"][:used, 0] >= 0
    lhs = float((f64(recv_x[:used][rows]) * f64(G[:used][rows])).sum())
    rhs = float((f64(x) * f64(gx)).sum())
    # grad_x is rounded once to bf16: relative 2^-9 per element
    bound = float((np.abs(f64(x)) * np.abs(f64(gx))).sum()) * 2.0**-8 + 1e-12
    assert abs(lhs - rhs) <= bound


def test_dispatch_backward_counts_selections():
    rng, idx, lay = _case(1)
    G = bf(np.ones((lay["cap"], 8)))
    gx, _ = oracle.dispatch_backward(G, lay["slot_of"])
    n = (idx >= 0).sum(axis=1)
    assert np.array_equal(f64(gx), np.repeat(n[:, None], 8, axis=1).astype(np.float64))


def test_dispatch_backward_weight_gradient_gather():
    rng, idx, lay = _case(2)
    gw_rows = rng.standard_normal(lay["cap"]).astype(np.float32)
    _, gw = oracle.dispatch_backward(bf(np.zeros((lay["cap"], 8))), lay["slot_of"], gw_rows)
    so = lay["slot_of"]
    assert np.array_equal(gw[so >= 0], gw_rows[so[so >= 0]])
    assert np.all(gw[so < 0] == 0)


def test_unweighted_combine_backward_is_dispatch():
    """The page's duality: the transpose of the unweighted combine is a
    dispatch -- grad_Y rows are bit copies of dy."""
    rng, idx, lay = _case(3)
    dy = bf(rng.standard_normal((idx.shape[0], 24)))
    gY, _ = oracle.combine_backward(dy, None, lay["slot_of"], lay["cap"], want_grad_w=False)
    ref, _ = oracle.dispatch_bf16(dy, None, lay)
    used = lay["expert_start"][-1]
    rows = lay["src_info"][:used, 0] >= 0
    assert np.array_equal(gY[:used][rows], ref[:used][rows])


def test_weighted_combine_backward_adjoint():
    rng, idx, lay = _case(4)
    T, H = idx.shape[0], 24
    w = rng.random((T, 3)).astype(np.float32)
    Y = bf(rng.standard_normal((lay["cap"], H)))
    dy = bf(rng.standard_normal((T, H)))
    y = oracle.combine(Y, w, lay["slot_of"])
    gY, gw = oracle.combine_backward(dy, w, lay["slot_of"], lay["cap"], Y)
    used = lay["expert_start"][-1]
    rows = lay["src_info"][:used, 0] >= 0
    lhs = float((f64(dy) * f64(y)).sum())
    rhs = float((f64(gY[:used][rows]) * f64(Y[:used][rows])).sum())
    bound = 2.0**-7 * float((np.abs(f64(dy)) * np.abs(f64(y))).sum()) + \
        2.0**-7 * float((np.abs(f64(gY[:used][rows])) * np.abs(f64(Y[:used][rows]))).sum())
    assert abs(lhs - rhs) <= bound
    # gate gradient: d<dy, y>/dw[t,k] = <dy_t, Y_slot>, exact in double
    so = lay["slot_of"]
    for t in range(T):
        for k in range(3):
            if so[t, k] < 0:
                assert gw[t, k] == 0
            else:
                want = float((f64(dy[t]) * f64(Y[so[t, k]])).sum())
                assert gw[t, k] == np.float32(want)


def test_backward_of_the_190_example(golden):
    g = dict(golden("worked_values.txt"))
    o = [float(v) for v in g["p4_outputs"]]
    gates = np.array([[float(v) for v in g["p4_gates"]]], np.float32)
    Y = bf([[o[0], o[1]], [o[2], o[3]]])
    so = np.array([[0, 1]], np.int32)
    dy = bf([[1.0, 1.0]])
    gY, gw = oracle.combine_backward(dy, gates, so, 2, Y)
    assert list(gw[0]) == [1.0, 4.0]               # <dy, (1,0)>, <dy, (4,0)>
    assert np.array_equal(gY[0], bf([[0.70, 0.70]])[0])
    assert np.array_equal(gY[1], bf([[0.30, 0.30]])[0])


def test_combine_backward_masked_and_padding_untouched():
    rng, idx, lay = _case(5, mask=0.4)
    dy = bf(rng.standard_normal((idx.shape[0], 8)))
    gY, gw = oracle.combine_backward(dy, None, lay["slot_of"], lay["cap"],
                                     bf(np.ones((lay["cap"], 8))), fill=0xABCD)
    assert np.all(gw[idx < 0] == 0)
    untouched = np.ones(lay["cap"], bool)
    untouched[lay["slot_of"][idx >= 0]] = False
    assert np.all(gY[untouched] == 0xABCD)
