"""Pins for the oracle's non-expanded (destination-major) stage: rank rows,
dispatch to ranks, expansion to expert rows, per-rank reduction and the
token-major sum over ranks.

Sources: "Deep Dive - DeepEP" ("Why expert parallelism needs a communication
layer": a token travels once per selected destination rank, an optional
expansion makes one slot per expert; "A four-token routing ledger" / "A
runnable routing ledger": rank 0 sends a to expert 3 and b to expert 2 and
receives c for expert 1 and d for expert 0; 8 vs 7 destination rows;
"Combine: reverse routing plus reduction": a bf16 local subtotal of 256 + 1
is 256 and the final result 0, against 1 for one final cast) and "GPU
Microarchitecture: DeepEP from First Principles" 2.1 / 1.2.
"""

import numpy as np

import oracle
import workloads
from workloads import to_bf16_bits


def bf(a):
    return to_bf16_bits(np.asarray(a, np.float32))


def _ledger(golden, variant=None):
    g = golden("routing_ledger.txt")
    gd = dict(g)
    names = [v[0] for k, v in g if k == "token"]
    routes = {v[0]: v[1:] for k, v in g if k == "route"}
    if variant:
        r = gd[variant]
        routes[r[0]] = r[1:]
    idx = np.array([[int(routes[n][0]), int(routes[n][2])] for n in names], np.int64)
    w = np.array([[float(routes[n][1]), float(routes[n][3])] for n in names], np.float32)
    return names, idx, w


def test_ledger_rank_rows(golden):
    names, idx, w = _ledger(golden)
    lay = oracle.layout(idx, 4, 2, 4)
    rl = oracle.rank_layout(lay)
    assert rl["rows"] == 8
    # rank 0 receives a, b (its own) and c, d; rank 1 the same four tokens
    r0 = [names[t] for t in rl["rank_src"][rl["rank_row_start"][0]:rl["rank_row_start"][1]]]
    r1 = [names[t] for t in rl["rank_src"][rl["rank_row_start"][1]:rl["rank_row_start"][2]]]
    assert r0 == ["a", "b", "c", "d"] and r1 == ["a", "b", "c", "d"]
    x = bf(np.arange(16).reshape(4, 4))
    _, ridx, rw = oracle.dispatch_ranks(x, idx, w, rl, 4)
    # local expert ids (expert - 2 * rank) in top-k order, -1 off the rank
    want = {("a", 0): [0, -1], ("b", 0): [-1, 1], ("c", 0): [1, -1], ("d", 0): [0, -1],
            ("a", 1): [-1, 1], ("b", 1): [0, -1], ("c", 1): [-1, 1], ("d", 1): [-1, 0]}
    for (n, r), ids in want.items():
        row = rl["rank_slot_of"][names.index(n), r]
        assert list(ridx[row]) == ids
        kept = np.array(ids) >= 0
        assert np.array_equal(rw[row][kept], w[names.index(n)][kept])
        assert np.all(rw[row][~kept] == 0)


def test_ledger_same_rank_seven_rows(golden):
    names, idx, w = _ledger(golden, "same_rank_route")
    lay = oracle.layout(idx, 4, 2, 4)
    rl = oracle.rank_layout(lay)
    assert rl["rows"] == 7
    a = names.index("a")
    assert rl["rank_slot_of"][a, 0] == -1
    _, ridx, _ = oracle.dispatch_ranks(bf(np.zeros((4, 2))), idx, w, rl, 4)
    assert list(ridx[rl["rank_slot_of"][a, 1]]) == [0, 1]   # experts 2 and 3


def test_rank_layout_invariants():
    rng = np.random.default_rng(0)
    T, E, K, R = 200, 32, 6, 8
    idx = workloads.random_routes(rng, T, E, K, mask_frac=0.2)
    lay = oracle.layout(idx, E, R, 8)
    rl = oracle.rank_layout(lay)
    assert np.array_equal(np.diff(rl["rank_row_start"]), lay["tokens_per_rank"])
    so = rl["rank_slot_of"]
    assert np.array_equal(so >= 0, lay["is_token_in_rank"] == 1)
    for r in range(R):
        seg = rl["rank_src"][rl["rank_row_start"][r]:rl["rank_row_start"][r + 1]]
        assert np.all(np.diff(seg) > 0)                  # token order
        assert np.array_equal(so[seg, r], np.arange(rl["rank_row_start"][r],
                                                     rl["rank_row_start"][r + 1]))


def test_expand_after_dispatch_to_ranks_is_the_expanded_dispatch():
    rng = np.random.default_rng(1)
    T, H, E, K, R = 64, 32, 16, 4, 4
    idx = workloads.random_routes(rng, T, E, K, mask_frac=0.15)
    lay = oracle.layout(idx, E, R, 4)
    rl = oracle.rank_layout(lay)
    x = bf(rng.standard_normal((T, H)))
    w = rng.random((T, K)).astype(np.float32)
    rank_x, _, rank_w = oracle.dispatch_ranks(x, idx, w, rl, E)
    ex, ew = oracle.expand(idx, lay, rl, rank_x, rank_w, E)
    dx, dw = oracle.dispatch_bf16(x, w, lay)
    used = lay["expert_start"][-1]
    rows = lay["src_info"][:used, 0] >= 0
    assert np.array_equal(ex[:used][rows], dx[:used][rows])
    assert np.array_equal(ew[:used][rows], dw[:used][rows])


def test_two_stage_reduction_cancellation(golden):
    """256 and 1 from two experts of rank 0, -256 from rank 1: the rank's bf16
    subtotal is 256 and the final result 0; one fp32 fold gives 1."""
    g = dict(golden("worked_values.txt"))
    a, b, c = [float(v) for v in g["p9_terms"]]
    idx = np.array([[0, 1, 2]], np.int64)                # E=4, R=2: ranks 0, 0, 1
    lay = oracle.layout(idx, 4, 2, 1)
    rl = oracle.rank_layout(lay)
    Y = np.zeros((lay["cap"], 1), np.uint16)
    Y[lay["slot_of"][0]] = bf([[a], [b], [c]])
    ry = oracle.reduce_ranks(idx, lay, rl, Y, None, 4)
    assert oracle.bf16_to_f32(ry[rl["rank_slot_of"][0, 0], 0]) == float(g["p9_local_subtotal"][0])
    y2 = oracle.combine_ranks(rl, ry)
    assert oracle.bf16_to_f32(y2[0, 0]) == float(g["p9_two_stages"][0])
    y1 = oracle.combine(Y, None, lay["slot_of"])
    assert oracle.bf16_to_f32(y1[0, 0]) == float(g["p9_single_stage"][0])


def test_two_stage_equals_one_stage_on_exact_values():
    rng = np.random.default_rng(2)
    T, H, E, K, R = 50, 8, 16, 4, 4
    idx = workloads.random_routes(rng, T, E, K, mask_frac=0.1)
    lay = oracle.layout(idx, E, R, 2)
    rl = oracle.rank_layout(lay)
    Y = bf(rng.integers(-8, 8, (lay["cap"], H)))        # small integers: sums exact
    w = np.ones((T, K), np.float32)
    ry = oracle.reduce_ranks(idx, lay, rl, Y, w, E)
    assert np.array_equal(oracle.combine_ranks(rl, ry), oracle.combine(Y, w, lay["slot_of"]))
