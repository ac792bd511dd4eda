"""Pins for the oracle's dispatch (bf16 copy, fused FP8) and combine.

Pinned against: the worked examples of "GPU Microarchitecture: DeepEP from
First Principles" 1.2 and of "Deep Dive - DeepEP" ("Combine: reverse routing
plus reduction", "A runnable routing ledger", "Precision: FP8 on the wire,
BF16 for the reduction"); identity reconstruction; the transpose relation of
dispatch and combine ("Deep Dive - DeepEP", backward duality in the combine
section); and the FP8 quantisation error bound.
"""

import numpy as np
import pytest

import oracle
import workloads
from workloads import to_bf16_bits


def bf(a):
    return to_bf16_bits(np.asarray(a, np.float32))


def f32(h):
    return oracle.bf16_to_f32_array(h)


def ulp_bf16(v):
    v = abs(float(v))
    if v == 0:
        return 2.0**-133
    e = np.floor(np.log2(v))
    return 2.0 ** (e - 7)


def run_layout(idx, E, R, A):
    lay = oracle.layout(np.asarray(idx, np.int64), E, R, A)
    assert lay["status"] == oracle.OK
    return lay


# ------------------------------------------------------------- worked values --

def test_p1_output_t0(golden):
    rows = [v for k, v in golden("worked_values.txt") if k == "p1_route"]
    idx = np.array([[int(r[1]), int(r[3])] for r in rows], np.int64)
    w = np.array([[0.73, 0.27], [0.6, 0.4], [0.5, 0.5]], np.float32)
    assert rows[0][2] == "0.73" and rows[0][4] == "0.27"
    E, H = 8, 8
    lay = run_layout(idx, E, 2, 1)
    x = bf(np.random.default_rng(0).standard_normal((3, H)))
    recv_x, _ = oracle.dispatch_bf16(x, w, lay)
    # identity metadata: the slot of (T0, k=0) lies in Expert2's segment and
    # maps back to token 0, selection 0
    s = lay["slot_of"][0, 0]
    assert lay["expert_start"][2] <= s < lay["expert_end"][2]
    assert tuple(lay["src_info"][s]) == (0, 0)
    # expert e multiplies by (e + 1); exact in bf16 for these small factors
    Y = np.zeros_like(recv_x)
    for e in range(E):
        a, b = lay["expert_start"][e], lay["expert_end"][e]
        Y[a:b] = bf(f32(recv_x[a:b]) * (e + 1))
    y = f32(oracle.combine(Y, w, lay["slot_of"]))
    x0 = f32(x[0]).astype(np.float64)
    want = 0.73 * 3 * x0 + 0.27 * 8 * x0
    for i in range(H):
        assert abs(y[0, i] - want[i]) <= ulp_bf16(want[i]) + 1e-6


def test_p4_weighted_once_raw_twice(golden):
    g = dict(golden("worked_values.txt"))
    o = [float(v) for v in g["p4_outputs"]]
    gates = np.array([[float(v) for v in g["p4_gates"]]], np.float32)
    Y = bf([[o[0], o[1]], [o[2], o[3]]])
    so = np.array([[0, 1]], np.int32)
    once = f32(oracle.combine(Y, gates, so))[0]
    raw = f32(oracle.combine(Y, None, so))[0]
    pre = bf(f32(Y) * gates.reshape(2, 1))
    twice = f32(oracle.combine(pre, gates, so))[0]
    for got, key in ((once, "p4_weighted_once"), (raw, "p4_unweighted"),
                     (twice, "p4_weighted_twice")):
        want = [float(v) for v in g[key]]
        for a, b in zip(got, want):
            assert abs(a - b) <= ulp_bf16(b) + 1e-6, (key, got, want)
    # caller-weighted rows into an unweighted combine give the same as once
    assert np.allclose(f32(oracle.combine(pre, None, so))[0], once, atol=0.02)


def test_p9_single_final_cast(golden):
    g = dict(golden("worked_values.txt"))
    terms = [float(v) for v in g["p9_terms"]]
    Y = bf([[t] for t in terms])
    so = np.array([[0, 1, 2]], np.int32)
    got = f32(oracle.combine(Y, None, so))[0, 0]
    assert got == float(g["p9_single_stage"][0])


def _ledger(golden, variant=None):
    g = golden("routing_ledger.txt")
    gd = dict(g)
    tok = [(v[0], int(v[1]), [float(v[2]), float(v[3])]) for k, v in g if k == "token"]
    names = [t[0] for t in tok]
    routes = {v[0]: v[1:] for k, v in g if k == "route"}
    if variant:
        r = gd[variant]
        routes[r[0]] = r[1:]
    idx = np.array([[int(routes[n][0]), int(routes[n][2])] for n in names], np.int64)
    w = np.array([[float(routes[n][1]), float(routes[n][3])] for n in names], np.float32)
    H = 8  # the page's 2 coordinates embedded in 8 channels, rest zero
    x = np.zeros((4, H), np.float32)
    for i, t in enumerate(tok):
        x[i, :2] = t[2]
    return gd, names, idx, w, bf(x)


def _ledger_run(idx, w, x, shuffle_seed=None):
    lay = run_layout(idx, 4, 2, 4)
    recv_x, recv_w = oracle.dispatch_bf16(x, w, lay, zero_padding=True)
    Y = np.zeros_like(recv_x)
    for e in range(4):
        a, b = lay["expert_start"][e], lay["expert_end"][e]
        Y[a:b] = bf(f32(recv_x[a:b]) * (e + 1))
    return lay, recv_w, Y


def test_p5_ledger_combined_rows(golden):
    gd, names, idx, w, x = _ledger(golden)
    lay, recv_w, Y = _ledger_run(idx, w, x)
    y = f32(oracle.combine(Y, w, lay["slot_of"]))
    for k, v in golden("routing_ledger.txt"):
        if k == "combined":
            i = names.index(v[0])
            for c in range(2):
                want = float(v[1 + c])
                # printed to 2 decimals; 1 bf16 ulp for the final cast
                assert abs(y[i, c] - want) <= ulp_bf16(want) + 0.005, (v, y[i])
    assert np.all(y[:, 2:] == 0)
    # received gate weights ride with their rows; padding rows carry 0
    so = lay["slot_of"]
    assert np.array_equal(recv_w[so.reshape(-1)], w.reshape(-1))
    pad = np.ones(lay["expert_start"][-1], bool)
    pad[so.reshape(-1)] = False
    assert np.all(recv_w[: lay["expert_start"][-1]][pad] == 0)


def test_p5_combine_ignores_row_order(golden):
    """Shuffling the expert rows (and the slot map with them) leaves the
    combined rows unchanged: combine follows the saved inverse map."""
    gd, names, idx, w, x = _ledger(golden)
    lay, _, Y = _ledger_run(idx, w, x)
    base = oracle.combine(Y, w, lay["slot_of"])
    perm = np.random.default_rng(5).permutation(Y.shape[0])
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    so = lay["slot_of"].copy()
    so[so >= 0] = inv[so[so >= 0]]
    assert np.array_equal(oracle.combine(Y[perm], w, so), base)


def test_p6_same_rank_value(golden):
    gd, names, idx, w, x = _ledger(golden, "same_rank_route")
    lay, _, Y = _ledger_run(idx, w, x)
    y = f32(oracle.combine(Y, w, lay["slot_of"]))
    want = float(gd["same_rank_combined_a_x"][0])
    assert abs(y[names.index("a"), 0] - want) <= ulp_bf16(want) + 0.005


def test_p7_masked_value_no_renormalisation(golden):
    gd, names, idx, w, x = _ledger(golden, "masked_route")
    lay, _, Y = _ledger_run(idx, w, x)
    y = f32(oracle.combine(Y, w, lay["slot_of"]))
    want = [float(v) for v in gd["masked_combined_a"]]
    for c in range(2):
        assert abs(y[names.index("a"), c] - want[c]) <= ulp_bf16(want[c]) + 1e-6


def test_p8_padding_never_gains_identity(golden):
    gd, names, idx, w, x = _ledger(golden)
    lay, _, Y = _ledger_run(idx, w, x)
    # poison every padding row: combine must not see it
    Y2 = Y.copy()
    for e in range(4):
        Y2[lay["expert_end"][e]: lay["expert_start"][e + 1]] = bf(999.0)
    assert np.array_equal(oracle.combine(Y2, w, lay["slot_of"]),
                          oracle.combine(Y, w, lay["slot_of"]))
    for e in range(4):
        assert np.all(lay["src_info"][lay["expert_end"][e]: lay["expert_start"][e + 1]] == -1)


# ---------------------------------------------------------- whole-path laws --

@pytest.mark.parametrize("name", ["tiny", "prefill"])
def test_identity_experts_reconstruct_input(name):
    wl = workloads.WORKLOADS[name]
    wl = wl.with_(num_tokens=min(wl.num_tokens, 256), hidden=min(wl.hidden, 512))
    inp = workloads.make_inputs(wl, seed=0)
    lay = run_layout(inp["topk_idx"], wl.num_experts, wl.num_ranks, 128)
    recv_x, _ = oracle.dispatch_bf16(inp["x"], inp["topk_weights"], lay)
    y = oracle.combine(recv_x, inp["topk_weights"], lay["slot_of"])
    # weights sum to 1 within a few fp32 ulps: far from any bf16 midpoint, so
    # y == x bit for bit, except that -0.0 comes back as +0.0 (the fold
    # starts from +0.0)
    x = inp["x"]
    assert np.array_equal(np.where(x == 0x8000, 0, x), y)


def test_dispatch_combine_duality():
    """<combine(Y; w=1), x> == <Y, dispatch(x)> up to the final bf16 cast."""
    rng = np.random.default_rng(7)
    T, H, E, K, R = 40, 16, 8, 3, 4
    idx = workloads.random_routes(rng, T, E, K, mask_frac=0.2)
    lay = run_layout(idx, E, R, 4)
    x = bf(rng.standard_normal((T, H)))
    Y = bf(rng.standard_normal((lay["cap"], H)))
    recv_x, _ = oracle.dispatch_bf16(x, None, lay, zero_padding=True)
    y = f32(oracle.combine(Y, None, lay["slot_of"])).astype(np.float64)
    xf, Yf = f32(x).astype(np.float64), f32(Y).astype(np.float64)
    used = lay["expert_start"][-1]
    lhs = float((y * xf).sum())
    rhs = float((Yf[:used] * f32(recv_x[:used]).astype(np.float64)).sum())
    bound = float((np.abs(y) * np.abs(xf)).sum()) * 2.0**-8 + 1e-9
    assert abs(lhs - rhs) <= bound


def test_zero_tokens_and_all_masked():
    lay = run_layout(np.zeros((0, 2), np.int64), 4, 2, 4)
    assert lay["expert_start"][-1] == 0
    x = np.zeros((0, 8), np.uint16)
    recv_x, _ = oracle.dispatch_bf16(x, None, lay)
    idx = np.full((3, 2), -1, np.int64)
    lay = run_layout(idx, 4, 2, 4)
    Y = bf(np.ones((4, 8)))
    y = oracle.combine(Y, np.ones((3, 2), np.float32), lay["slot_of"])
    assert np.all(y == 0)      # +0.0, not -0.0


# -------------------------------------------------------------------- FP8 ---

def test_p11_fp8_row_bytes(golden):
    H, q_bytes, s_bytes, bf_bytes = [int(v) for v in dict(golden("worked_values.txt"))["p11_row"]]
    idx = np.array([[0]], np.int64)
    lay = run_layout(idx, 1, 1, 1)
    x = bf(np.random.default_rng(0).standard_normal((1, H)))
    q, s, _ = oracle.dispatch_fp8(x, None, lay)
    assert q[0].nbytes == q_bytes and s[0].nbytes == s_bytes
    assert x[0].nbytes == bf_bytes


def test_fp8_quantisation_error_bound():
    rng = np.random.default_rng(11)
    T, H = 64, 512
    xs = rng.standard_normal((T, H)) * np.exp(rng.uniform(-8, 8, (T, 1)))
    x = bf(xs)
    idx = np.arange(T, dtype=np.int64).reshape(T, 1) % 8
    lay = run_layout(idx, 8, 2, 1)
    q, s, _ = oracle.dispatch_fp8(x, None, lay)
    xf = f32(x).astype(np.float64)
    for t in range(T):
        slot = lay["slot_of"][t, 0]
        deq = oracle.e4m3_to_f32_array(q[slot]).astype(np.float64)
        sc = np.repeat(s[slot].astype(np.float64), 128)
        v = xf[t] / sc
        half_ulp = np.where(np.abs(v) >= 2.0**-6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 1e-300))) - 4), 2.0**-10)
        err = np.abs(deq * sc - xf[t])
        assert np.all(err <= (half_ulp + np.abs(v) * 2.0**-23) * sc * (1 + 2.0**-20))
        # the block maximum maps to (nearly) 448
        for c in range(H // 128):
            blk = np.abs(xf[t, c * 128:(c + 1) * 128])
            assert s[slot, c] == np.float32(np.float32(blk.max()) / np.float32(448.0))
            assert np.max(np.abs(deq[c * 128:(c + 1) * 128])) == 448.0


def test_fp8_zero_block_and_padding():
    H = 256
    x = np.zeros((2, H), np.uint16)
    x[1, 128:] = bf(np.linspace(-3, 3, 128))
    idx = np.array([[0], [0]], np.int64)
    lay = run_layout(idx, 2, 1, 4)
    q, s, w = oracle.dispatch_fp8(x, np.ones((2, 1), np.float32), lay, zero_padding=True)
    assert np.all(q[0] == 0) and np.all(s[0] == 0)
    assert s[1, 0] == 0 and np.all(q[1, :128] == 0) and s[1, 1] > 0
    assert np.all(q[2:4] == 0) and np.all(s[2:4] == 0) and np.all(w[2:4] == 0)


def test_fp8_each_copy_identical():
    rng = np.random.default_rng(2)
    T, H, E, K = 16, 384, 8, 4
    idx = workloads.random_routes(rng, T, E, K)
    lay = run_layout(idx, E, 4, 2)
    x = bf(rng.standard_normal((T, H)))
    q, s, _ = oracle.dispatch_fp8(x, None, lay)
    for t in range(T):
        slots = lay["slot_of"][t]
        for sl in slots[1:]:
            assert np.array_equal(q[sl], q[slots[0]]) and np.array_equal(s[sl], s[slots[0]])
