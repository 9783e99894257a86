"""Pins of the oracle's expert-parallel index functions (CPU only), and the
library's host-side EPLB plan against the oracle's.

What they restate: the dispatch and combine of expert parallelism
(Awesome-ML-SYS-Tutorial MoE/EP guide, gsyq.cn, "Expert Parallelism": split
sizes from per-expert counts, all-to-all, the receiver's re-sort of its
chunks by local expert, combine by all-to-all; hotspot experts and EPLB-style
replication).
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("A,B,seed", [(1, 1, 0), (3, 5, 1), (8, 8, 2), (4, 64, 3), (16, 3, 4)])
def test_sort_chunks_is_a_chunk_transpose(A, B, seed):
    """Pin: against an independent formulation (a lexsort of every input
    row's key (b, a, position in its chunk)); transposing back with the
    transposed counts restores the input order; group offsets are the
    cumulative column sums."""
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 5, size=(A, B))
    counts[rng.random((A, B)) < 0.3] = 0            # empty chunks
    src_of, pos_of, group = oracle.sort_chunks(counts)
    N = int(counts.sum())
    a_of, b_of, l_of = [], [], []
    for a in range(A):
        for b in range(B):
            for l in range(counts[a, b]):
                a_of.append(a), b_of.append(b), l_of.append(l)
    order = np.lexsort((np.array(l_of), np.array(a_of), np.array(b_of))) if N else np.zeros(0, int)
    np.testing.assert_array_equal(src_of, order)
    np.testing.assert_array_equal(pos_of[src_of], np.arange(N))
    np.testing.assert_array_equal(group, np.concatenate([[0], np.cumsum(counts.sum(0))]))
    back_src, _, _ = oracle.sort_chunks(counts.T)   # output rows are in (b, a) chunks
    np.testing.assert_array_equal(src_of[back_src], np.arange(N))


def test_map_replicas_sends_each_row_to_a_replica_of_its_expert():
    """Pin: every assignment goes to a physical expert of its own logical
    expert, to replica t mod replicas (checked by the formula, row by row),
    and an expert with one replica keeps its rows."""
    rng = np.random.default_rng(5)
    T, k, E = 50, 3, 6
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    plan = oracle.eplb_plan(np.bincount(ids.reshape(-1), minlength=E), 2, 10)
    phys = oracle.map_replicas(ids, plan["rep_first"], plan["rep_count"], plan["rep_list"])
    np.testing.assert_array_equal(plan["phys_to_log"][phys], ids)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            r = list(plan["rep_list"][plan["rep_first"][e]:plan["rep_first"][e] + plan["rep_count"][e]]).index(phys[t, j])
            assert r == t % plan["rep_count"][e]


def test_eplb_plan_hand_case():
    """Pin: a case worked by hand (tests/golden/eplb_hand_case.json)."""
    g = json.load(open(os.path.join(GOLDEN, "eplb_hand_case.json")))
    plan = oracle.eplb_plan(g["load"], g["G"], g["n_phys"])
    for key in ("phys_to_log", "rep_first", "rep_count", "rep_list", "rank_load"):
        np.testing.assert_array_equal(plan[key], g[key], err_msg=key)


@pytest.mark.parametrize("E,G,extra,seed", [(8, 2, 0, 0), (8, 4, 4, 1), (16, 4, 8, 2), (128, 8, 16, 3)])
def test_eplb_plan_invariants(E, G, extra, seed):
    """Pin: every expert has a replica, replicas fill the physical slots, each
    rank holds n_phys / G of them, the tables agree, the rank loads sum to
    the total, and each extra replica went to the expert with the largest
    load per replica at that point (brute force)."""
    rng = np.random.default_rng(seed)
    load = (rng.zipf(1.3, size=E) * 17 % 5000).astype(np.int64)
    n_phys = E + extra
    plan = oracle.eplb_plan(load, G, n_phys)
    rc = plan["rep_count"]
    assert rc.min() >= 1 and rc.sum() == n_phys
    assert sorted(plan["rep_list"].tolist()) == list(range(n_phys))
    for e in range(E):
        for r in range(rc[e]):
            assert plan["phys_to_log"][plan["rep_list"][plan["rep_first"][e] + r]] == e
    assert plan["rank_load"].sum() == load.sum()
    rep = np.ones(E, np.int64)
    for _ in range(extra):
        ratio = [load[e] / rep[e] for e in range(E)]
        best = int(np.argmax(ratio))                 # the first maximum: the lower index on ties
        rep[best] += 1
    np.testing.assert_array_equal(rc, rep)
    per_rank = np.bincount(np.arange(n_phys) // (n_phys // G), minlength=G)
    assert (per_rank == n_phys // G).all()


def test_eplb_plan_splits_a_hotspot():
    """Special case: one expert with 100x the load of each other one, on 4
    ranks.  Without replicas its rank carries it alone (1010); with four extra
    replicas it is split five ways (200 rows each), one rank takes two of
    them, and the busiest rank drops to 410 (worked by hand: the four ranks
    take one replica each, the fifth goes to rank 0 on the tie, then the 10s
    go to ranks 1-3 first)."""
    load = [1000] + [10] * 7
    base = oracle.eplb_plan(load, 4, 8)
    plan = oracle.eplb_plan(load, 4, 12)
    assert base["rank_load"].max() == 1010
    assert plan["rep_count"][0] == 5
    np.testing.assert_array_equal(plan["rank_load"], [410, 220, 220, 220])


@pytest.mark.parametrize("E,G,extra,seed", [(8, 2, 2, 0), (16, 4, 8, 1), (128, 8, 24, 2), (256, 16, 0, 3)])
def test_library_eplb_plan_equals_oracle(E, G, extra, seed):
    """The library's host-side moe_eplb_plan (C++) gives the oracle's plan exactly."""
    import token_dispatch_grouped_softmax_gb300 as moe

    rng = np.random.default_rng(seed)
    load = rng.integers(0, 3000, size=E)
    load[rng.random(E) < 0.2] = 0
    got = moe.ops.eplb_plan(load, G, E + extra)
    ref = oracle.eplb_plan(load, G, E + extra)
    for key in ref:
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_ep_dispatch_is_the_local_permutation(G):
    """Pin: the rows each rank's experts receive, in order, are exactly the
    local (non-EP) permutation's rows of those experts when the sources hold
    consecutive token ranges; G = 1 is the local permutation itself."""
    rng = np.random.default_rng(G)
    T, k, E = 37, 2, 8
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    sizes = [T // G + (1 if s < T % G else 0) for s in range(G)]
    starts = np.concatenate([[0], np.cumsum(sizes)])
    per_rank = [ids[starts[s]:starts[s + 1]] for s in range(G)]
    got = oracle.ep_dispatch(per_rank, E, G)
    local = oracle.permute(ids, E)
    P = E // G
    for d, (rows, offs) in enumerate(got):
        tokens = [starts[s] + t for s, t, j in rows]
        want = local["src_row"][local["offsets"][d * P]:local["offsets"][(d + 1) * P]]
        np.testing.assert_array_equal(tokens, want)
        np.testing.assert_array_equal(offs, local["offsets"][d * P:(d + 1) * P + 1] - local["offsets"][d * P])
        for (s, t, j) in rows:
            assert d * P <= per_rank[s][t, j] < (d + 1) * P
