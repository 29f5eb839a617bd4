"""Pins for the oracle's best-first tree (CPU only).

What fixes the answer: the hand-worked example in tests/golden, brute-force
enumeration of every lattice path sorted by the recursive total order, the
structural invariants of a best-first tree, and the two degenerate lattices
(K = 1 gives a chain, m = 1 gives a star in rank order).
"""
import json
import os

import numpy as np
import pytest

import oracle
from tests.indep import brute_force_tree, canonical_order

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_tree():
    g = json.load(open(os.path.join(GOLD, "tree_hand_example.json")))
    tok = np.array([g["lat_tok"]], np.int32)
    sc = np.array([g["lat_score"]], np.float32)
    t = oracle.tree_build(tok, sc, np.array([g["root_tok"]], np.int32), g["N"])
    e = g["expect"]
    for key in ("node_tok", "node_parent", "node_depth", "node_rank"):
        assert t[key][0].tolist() == e[key], key
    assert t["node_score"][0].tolist() == e["node_score"]
    assert t["node_anc"][0, :, 0].tolist() == e["node_anc"]
    assert int(t["n_nodes"][0]) == e["n_nodes"]


def _lattice(rng, m, K, V=50, ties=False):
    tok = np.stack([rng.permutation(V)[:K] for _ in range(m)]).astype(np.int32)
    if ties:
        sc = -0.5 * rng.integers(0, 4, size=(m, K)).astype(np.float32)
    else:
        z = rng.normal(0, 2, size=(m, K))
        z = z - z.max(axis=1, keepdims=True)
        sc = (z - np.log(np.exp(z).sum(axis=1, keepdims=True))).astype(np.float32)
        sc = np.minimum(sc, np.float32(0))
    return tok, sc


@pytest.mark.parametrize("ties", [False, True])
def test_best_first_equals_brute_force(ties):
    rng = np.random.default_rng(1234 + ties)
    for trial in range(600):
        m = int(rng.integers(1, 5))
        K = int(rng.integers(1, 5))
        total = sum(K ** d for d in range(1, m + 1))
        N = int(rng.integers(0, min(total + 3, 127) + 1))
        tok, sc = _lattice(rng, m, K, ties=ties)
        root = int(rng.integers(0, 50))
        t = oracle.tree_build(tok[None], sc[None], np.array([root], np.int32), N)
        bf = brute_force_tree(tok, sc, root, N)
        assert int(t["n_nodes"][0]) == bf["n_nodes"] == 1 + min(N, total)
        for key in ("node_tok", "node_parent", "node_depth", "node_rank", "node_score"):
            np.testing.assert_array_equal(t[key][0], bf[key], err_msg=f"{key} trial {trial}")
        np.testing.assert_array_equal(t["node_anc"][0], bf["node_anc"])


def _check_invariants(t, tok, sc, m, K, N, root):
    n = int(t["n_nodes"])
    total = sum(K ** d for d in range(1, m + 1))
    assert n == 1 + min(N, total)
    par, dep, rank = t["node_parent"], t["node_depth"], t["node_rank"]
    score, ntok, anc = t["node_score"], t["node_tok"], t["node_anc"]
    assert ntok[0] == root and par[0] == -1 and dep[0] == 0 and score[0] == 0.0
    orders = [canonical_order(sc[s]) for s in range(m)]
    seen = set()
    for x in range(1, n):
        p = par[x]
        assert 0 <= p < x                              # parent precedes child
        assert dep[x] == dep[p] + 1 and 1 <= dep[x] <= m
        assert score[x] <= score[x - 1]                # best-first order
        s = dep[x] - 1
        assert ntok[x] == tok[s][orders[s][rank[x]]]
        assert score[x] == np.float32(score[p] + sc[s][orders[s][rank[x]]])
        assert (p, rank[x]) not in seen                # no duplicate edge
        seen.add((p, rank[x]))
        want = anc[p].copy()
        want[x // 64] |= np.uint64(1) << np.uint64(x % 64)
        np.testing.assert_array_equal(anc[x], want)
    for x in range(n, N + 1):                          # padding rows
        assert ntok[x] == -1 and par[x] == -1 and dep[x] == -1 and rank[x] == -1
        assert not anc[x].any()


@pytest.mark.parametrize("m,K,N", [(8, 16, 24), (16, 16, 64), (8, 16, 127), (3, 2, 20)])
def test_invariants_at_workload_shapes(m, K, N):
    rng = np.random.default_rng(m * 1000 + N)
    for _ in range(20):
        tok, sc = _lattice(rng, m, K, V=151936)
        root = int(rng.integers(0, 151936))
        t = oracle.tree_build(tok[None], sc[None], np.array([root], np.int32), N)
        _check_invariants({k: v[0] for k, v in t.items()}, tok, sc, m, K, N, root)


def test_k1_is_a_chain():
    rng = np.random.default_rng(7)
    for m in (1, 3, 8):
        for N in (0, 2, 5, 12):
            tok, sc = _lattice(rng, m, 1)
            t = oracle.tree_build(tok[None], sc[None], np.array([3], np.int32), N)
            n = int(t["n_nodes"][0])
            assert n == 1 + min(N, m)
            assert t["node_parent"][0, :n].tolist() == list(range(-1, n - 1))
            assert t["node_tok"][0, 1:n].tolist() == tok[: n - 1, 0].tolist()


def test_m1_is_a_star_in_rank_order():
    rng = np.random.default_rng(8)
    for K in (1, 4, 16):
        for N in (0, 3, 16, 20):
            tok, sc = _lattice(rng, 1, K)
            t = oracle.tree_build(tok[None], sc[None], np.array([3], np.int32), N)
            n = int(t["n_nodes"][0])
            assert n == 1 + min(N, K)
            assert (t["node_parent"][0, 1:n] == 0).all()
            assert t["node_rank"][0, 1:n].tolist() == list(range(n - 1))
            order = canonical_order(sc[0])
            assert t["node_tok"][0, 1:n].tolist() == [int(tok[0][order[r]]) for r in range(n - 1)]


def test_all_equal_scores_give_breadth_first_order():
    m, K, N = 3, 2, 14
    tok = np.arange(m * K, dtype=np.int32).reshape(m, K)
    sc = np.zeros((m, K), np.float32)
    t = oracle.tree_build(tok[None], sc[None], np.array([99], np.int32), N)
    # equal keys fall back to depth, then parent index, then rank: BFS
    assert t["node_depth"][0].tolist() == [0, 1, 1, 2, 2, 2, 2, 3, 3, 3, 3, 3, 3, 3, 3]
    assert t["node_parent"][0].tolist() == [-1, 0, 0, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5, 6, 6]


def test_batch_rows_are_independent():
    rng = np.random.default_rng(9)
    toks, scs = zip(*[_lattice(rng, 4, 4) for _ in range(3)])
    tok, sc = np.stack(toks), np.stack(scs)
    root = np.array([1, 2, 3], np.int32)
    t = oracle.tree_build(tok, sc, root, 10)
    for b in range(3):
        tb = oracle.tree_build(tok[b:b + 1], sc[b:b + 1], root[b:b + 1], 10)
        for key in t:
            np.testing.assert_array_equal(t[key][b], tb[key][0])


def test_duplicate_tokens_rejected():
    tok = np.array([[[1, 1]]], np.int32)
    sc = np.array([[[-1.0, -2.0]]], np.float32)
    with pytest.raises(ValueError):
        oracle.tree_build(tok, sc, np.array([0], np.int32), 2)
