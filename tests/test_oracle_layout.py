"""Pins for the oracle's layout (counts, aligned offsets, slots, identity
metadata, per-rank dedup).

Pinned against: the worked values of "GPU Microarchitecture: DeepEP from First
Principles" 6.1 and "Deep Dive - DeepEP" ("Dispatch: layout, move, and
epilogue"; "A runnable routing ledger"); brute force over every route of tiny
problems against a second, dictionary-based definition written from the
ledger's dispatch semantics; structural invariants; and the balanced-gate
closed form of "Deep Dive - DeepEP", "Analytical SM and QP sizing".
"""

import itertools
import math

import numpy as np
import pytest

import oracle
import workloads


# ---------------------------------------------------------------- helpers ---

def ledger_layout(routes, E, R, A):
    """Independent definition in the style of the page's routing ledger: walk
    tokens in order, append each selected (token, k) to its expert's list,
    pad every list to a multiple of A with empty rows, and concatenate the
    lists in expert order.  Returns (rows, counts, rank_rows)."""
    per_rank = E // R
    recv = {e: [] for e in range(E)}
    rank_rows = set()
    for t, choices in enumerate(routes):
        for k, e in enumerate(choices):
            if e == -1:
                continue
            rank_rows.add((t, e // per_rank))
            recv[e].append((t, k))
    counts = [len(recv[e]) for e in range(E)]
    rows = []
    for e in range(E):
        rows.extend(recv[e])
        rows.extend([(-1, -1)] * (-len(recv[e]) % A))
    return rows, counts, rank_rows


def check_invariants(lay, idx, E, R, A):
    T, K = idx.shape
    es, ee, cnt = lay["expert_start"], lay["expert_end"], lay["expert_count"]
    n = int((idx >= 0).sum())
    assert cnt.sum() == n
    assert es[0] == 0
    assert np.all(es[:-1] % A == 0) and es[-1] % A == 0
    assert np.array_equal(ee - es[:-1], cnt)
    assert np.all(ee <= es[1:])
    assert np.array_equal(lay["rank_start"], es[:: E // R])
    so = lay["slot_of"]
    assert np.array_equal(so < 0, idx < 0)
    used = so[so >= 0]
    assert np.unique(used).size == used.size == n          # bijection
    si = lay["src_info"]
    tt, kk = np.nonzero(so >= 0)
    assert np.array_equal(si[so[tt, kk], 0], tt)
    assert np.array_equal(si[so[tt, kk], 1], kk)
    # every slot sits inside its expert's valid range
    e_of = idx[tt, kk]
    assert np.all(so[tt, kk] >= es[e_of]) and np.all(so[tt, kk] < ee[e_of])
    # rows that carry no token are marked (-1, -1), padding included
    mask = np.ones(es[-1], bool)
    mask[used] = False
    assert np.all(si[: es[-1]][mask] == -1)
    # order within an expert: source-global (token, k) order
    for e in range(E):
        seg = si[es[e]: ee[e]]
        key = seg[:, 0].astype(np.int64) * K + seg[:, 1]
        assert np.all(np.diff(key) > 0)


# ------------------------------------------------------------- worked values --

def test_p2_unaligned_offsets(golden):
    g = golden("worked_values.txt")
    counts = [int(v) for v in dict(g)["p2_counts"]]
    E = len(counts)
    # one token per selection of a K=1 route with these counts
    idx = np.array([[e] for e in range(E) for _ in range(counts[e])], np.int64)
    lay = oracle.layout(idx, E, 1, 1)
    assert lay["status"] == oracle.OK
    for key, (e, off) in [(k, v) for k, v in g if k == "p2_offset"]:
        assert lay["expert_start"][int(e)] == int(off)
    assert list(lay["expert_count"]) == counts


def test_p3_alignment_psum(golden):
    g = dict(golden("worked_values.txt"))
    counts = [int(v) for v in g["p3_counts"]]
    A = int(g["p3_alignment"][0])
    idx = np.array([[e] for e in range(len(counts)) for _ in range(counts[e])], np.int64)
    lay = oracle.layout(idx, len(counts), 1, A)
    assert list(lay["expert_start"][:-1]) == [int(v) for v in g["p3_starts"]]
    assert list(lay["expert_end"]) == [int(v) for v in g["p3_ends"]]
    assert lay["expert_start"][-1] == int(g["p3_allocated"][0])
    assert list(lay["expert_count"]) == counts   # the unaligned counts


def _ledger_fixture(golden):
    g = golden("routing_ledger.txt")
    names = [v[0] for k, v in g if k == "token"]
    routes = {v[0]: v[1:] for k, v in g if k == "route"}
    idx = np.array([[int(routes[n][0]), int(routes[n][2])] for n in names], np.int64)
    return g, names, idx


def test_p5_ledger_expert_order(golden):
    g, names, idx = _ledger_fixture(golden)
    lay = oracle.layout(idx, 4, 2, 4)
    assert lay["status"] == oracle.OK
    es, ee, si = lay["expert_start"], lay["expert_end"], lay["src_info"]
    for k, v in g:
        if k == "order":
            e = int(v[0])
            got = [names[t] for t in si[es[e]: ee[e], 0]]
            assert got == v[1:]
    gd = dict(g)
    assert int((lay["slot_of"] >= 0).sum()) == int(gd["expert_slots"][0])
    assert int(es[-1]) == int(gd["allocated_slots"][0])
    assert int(lay["is_token_in_rank"].sum()) == int(gd["destination_rows"][0])
    check_invariants(lay, idx, 4, 2, 4)


def test_p6_same_rank_dedup(golden):
    g, names, idx = _ledger_fixture(golden)
    gd = dict(g)
    r = gd["same_rank_route"]
    idx[names.index(r[0])] = [int(r[1]), int(r[3])]
    lay = oracle.layout(idx, 4, 2, 4)
    assert int((lay["slot_of"] >= 0).sum()) == int(gd["same_rank_expert_slots"][0])
    assert int(lay["is_token_in_rank"].sum()) == int(gd["same_rank_destination_rows"][0])
    assert int(lay["tokens_per_rank"].sum()) == int(gd["same_rank_destination_rows"][0])


def test_p7_masked_selection(golden):
    g, names, idx = _ledger_fixture(golden)
    gd = dict(g)
    r = gd["masked_route"]
    idx[names.index(r[0])] = [int(r[1]), int(r[3])]
    lay = oracle.layout(idx, 4, 2, 4)
    assert int((lay["slot_of"] >= 0).sum()) == int(gd["masked_expert_slots"][0])
    assert int(lay["is_token_in_rank"].sum()) == int(gd["masked_destination_rows"][0])
    # -1 is "unused": never expert E-1
    assert lay["expert_count"][3] == 1          # only c, not a's masked slot
    check_invariants(lay, idx, 4, 2, 4)


def test_p12_range_and_duplicates():
    idx = np.array([[0, 1], [2, -1]], np.int64)
    assert oracle.layout(idx, 4, 2, 4)["status"] == oracle.OK
    for bad in (-2, 4, 100):
        b = idx.copy()
        b[1, 1] = bad
        assert oracle.layout(b, 4, 2, 4)["status"] == oracle.ERR_EXPERT_RANGE
    d = np.array([[1, 1]], np.int64)
    assert oracle.layout(d, 4, 2, 4)["status"] == oracle.ERR_DUP_EXPERT
    # two masked slots are not duplicates
    assert oracle.layout(np.array([[-1, -1]], np.int64), 4, 2, 4)["status"] == oracle.OK


def test_capacity_formula_is_worst_case():
    # every expert one row past a multiple of A: the padding bound is reached
    E, A, K = 4, 4, 1
    T = E * (A + 1)
    idx = np.array([[e] for e in range(E) for _ in range(A + 1)], np.int64)
    lay = oracle.layout(idx, E, 2, A)
    assert lay["expert_start"][-1] == E * 2 * A
    assert oracle.recv_capacity(T, K, E, A) >= lay["expert_start"][-1]
    assert oracle.recv_capacity(T, K, E, A) == T * K + E * (A - 1)


# -------------------------------------------------------------- brute force --

def _all_token_routes(E, K):
    opts = [-1] + list(range(E))
    out = []
    for combo in itertools.product(opts, repeat=K):
        sel = [c for c in combo if c >= 0]
        if len(sel) == len(set(sel)):
            out.append(combo)
    return out


@pytest.mark.parametrize("E,K,T_max", [(2, 1, 3), (4, 1, 3), (2, 2, 3), (4, 2, 2), (3, 2, 2)])
def test_brute_force_against_ledger_definition(E, K, T_max):
    per_tok = _all_token_routes(E, K)
    ranks = [r for r in (1, 2, 4) if E % r == 0]
    for T in range(0, T_max + 1):
        for routes in itertools.product(per_tok, repeat=T):
            idx = np.array(routes, np.int64).reshape(T, K)
            for A in (1, 2, 4):
                for R in ranks:
                    lay = oracle.layout(idx, E, R, A)
                    assert lay["status"] == oracle.OK
                    rows, counts, rank_rows = ledger_layout(routes, E, R, A)
                    used = int(lay["expert_start"][-1])
                    assert used == len(rows)
                    assert [tuple(r) for r in lay["src_info"][:used]] == rows
                    assert list(lay["expert_count"]) == counts
                    got = {(t, r) for t in range(T) for r in range(R)
                           if lay["is_token_in_rank"][t, r]}
                    assert got == rank_rows
                    assert int(lay["tokens_per_rank"].sum()) == len(rank_rows)
                    for t in range(T):
                        for k in range(K):
                            s = lay["slot_of"][t, k]
                            if routes[t][k] == -1:
                                assert s == -1
                            else:
                                assert rows[s] == (t, k)


# --------------------------------------------------------------- invariants --

@pytest.mark.parametrize("name", ["tiny", "skew", "prefill"])
def test_invariants_on_workloads(name):
    wl = workloads.WORKLOADS[name]
    if wl.num_tokens > 4096:
        wl = wl.with_(num_tokens=2048)
    inp = workloads.make_inputs(wl, seed=0)
    idx = inp["topk_idx"]
    lay = oracle.layout(idx, wl.num_experts, wl.num_ranks, wl.expert_alignment)
    assert lay["status"] == oracle.OK
    check_invariants(lay, idx, wl.num_experts, wl.num_ranks, wl.expert_alignment)


def test_masked_fraction_of_skew_workload():
    wl = workloads.WORKLOADS["skew"]
    inp = workloads.make_inputs(wl, seed=0)
    n_masked = int((inp["topk_idx"] < 0).sum())
    assert n_masked == round(0.05 * wl.num_tokens * wl.num_topk) == 2458
    lay = oracle.layout(inp["topk_idx"], wl.num_experts, wl.num_ranks, 128)
    assert int(lay["expert_count"].sum()) == 46694


# ------------------------------------------------------- balanced-gate law --

def expected_destinations(E, G, k):
    return G * (1 - math.comb(E - E // G, k) / math.comb(E, k))


def test_p10_closed_form_by_enumeration(golden):
    E, G, k, want = [float(v) for v in dict(golden("worked_values.txt"))["p10_case"]]
    E, G, k = int(E), int(G), int(k)
    pairs = list(itertools.combinations(range(E), k))
    enum = sum(len({e // (E // G) for e in p}) for p in pairs) / len(pairs)
    assert abs(enum - want) < 1e-6
    assert abs(expected_destinations(E, G, k) - enum) < 1e-12


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "sweep1k"])
def test_p10_mean_destinations_statistical(name):
    """Mean distinct destination ranks per token (the oracle's dedup) against
    the balanced-gate closed form, within 4 standard errors."""
    wl = workloads.WORKLOADS[name]
    T = max(wl.num_tokens, 2048)
    wl = wl.with_(num_tokens=T, hidden=8 if not wl.use_fp8_dispatch else 128)
    inp = workloads.make_inputs(wl, seed=3)
    lay = oracle.layout(inp["topk_idx"], wl.num_experts, wl.num_ranks, 128)
    d = lay["is_token_in_rank"].sum(axis=1).astype(np.float64)
    want = expected_destinations(wl.num_experts, wl.num_ranks, wl.num_topk)
    se = d.std(ddof=1) / math.sqrt(T)
    assert abs(d.mean() - want) <= 4 * se + 1e-9, (d.mean(), want, se)
