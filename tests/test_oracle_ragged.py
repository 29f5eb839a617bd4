"""Pins for the oracle's batch of trees sharing a node budget (CPU only).

The digest's batching mechanism (technical novelty) shares one node budget
across the batch (the target GEMM's 192-node plateau) and picks the number of
draft positions per request (16/12/8).  Reading: draft nodes are inserted
best-first over all requests' frontiers together, at most N per request.

What fixes the answer: brute force over tiny lattices (every path of every
request, globally sorted, taken greedily under the caps), the reduction to
independent best-first trees when there is no budget, and the budget and
depth invariants at workload shapes.
"""
import numpy as np
import pytest

import oracle
from tests.indep import brute_force_ragged


def _batch(rng, B, m, K, V=60, ties=False):
    tok = np.stack([np.stack([rng.permutation(V)[:K] for _ in range(m)]) for _ in range(B)]).astype(np.int32)
    if ties:
        sc = -0.5 * rng.integers(0, 4, size=(B, m, K)).astype(np.float32)
    else:
        z = rng.normal(0, 2, size=(B, m, K))
        z = z - z.max(axis=2, keepdims=True)
        sc = np.minimum((z - np.log(np.exp(z).sum(axis=2, keepdims=True))).astype(np.float32),
                        np.float32(0))
    return tok, sc


@pytest.mark.parametrize("ties", [False, True])
def test_shared_budget_equals_brute_force(ties):
    rng = np.random.default_rng(77 + ties)
    for trial in range(300):
        B = int(rng.integers(1, 4))
        m = int(rng.integers(1, 4))
        K = int(rng.integers(1, 4))
        N = int(rng.integers(0, 20))
        m_req = rng.integers(1, m + 1, size=B).astype(np.int32)
        budget = int(rng.integers(-1, B * N + 3))
        tok, sc = _batch(rng, B, m, K, ties=ties)
        root = rng.integers(0, 60, size=B).astype(np.int32)
        t = oracle.tree_build_ragged(tok, sc, root, N, m_req, budget)
        bf = brute_force_ragged(tok, sc, root, N, m_req, budget)
        for key in ("n_nodes", "node_tok", "node_parent", "node_depth", "node_rank", "node_anc"):
            np.testing.assert_array_equal(t[key], bf[key], err_msg=f"{key} trial {trial}")
        # keys compared bit for bit (a -0.0 edge must give a +0.0 key: 0 + edge)
        np.testing.assert_array_equal(t["node_score"].view(np.uint32),
                                      bf["node_score"].view(np.uint32), err_msg=f"score bits {trial}")


def test_no_budget_is_independent_trees_over_truncated_lattices():
    rng = np.random.default_rng(5)
    B, m, K, N = 4, 8, 16, 24
    tok, sc = _batch(rng, B, m, K, V=151936)
    root = rng.integers(0, 151936, size=B).astype(np.int32)
    m_req = np.array([8, 6, 3, 1], np.int32)
    t = oracle.tree_build_ragged(tok, sc, root, N, m_req, -1)
    for b in range(B):
        ref = oracle.tree_build(tok[b:b + 1, : m_req[b]], sc[b:b + 1, : m_req[b]], root[b:b + 1], N)
        for key in ref:
            np.testing.assert_array_equal(t[key][b:b + 1], ref[key], err_msg=f"{key} request {b}")
    full = oracle.tree_build_ragged(tok, sc, root, N, np.full(B, m, np.int32), -1)
    ref = oracle.tree_build(tok, sc, root, N)
    for key in ref:
        np.testing.assert_array_equal(full[key], ref[key])


@pytest.mark.parametrize("budget", [0, 1, 50, 96, 192, 1000])
def test_budget_and_depth_invariants(budget):
    rng = np.random.default_rng(budget + 3)
    B, m, K, N = 24, 16, 16, 24
    tok, sc = _batch(rng, B, m, K, V=151936)
    root = rng.integers(0, 151936, size=B).astype(np.int32)
    m_req = np.array([16, 12, 8] * 8, np.int32)
    t = oracle.tree_build_ragged(tok, sc, root, N, m_req, budget)
    drafts = t["n_nodes"] - 1
    assert drafts.sum() == min(budget, B * N)            # every lattice here has > N paths
    assert (drafts <= N).all()
    cut = []
    for b in range(B):
        n = int(t["n_nodes"][b])
        dep, par, score = t["node_depth"][b], t["node_parent"][b], t["node_score"][b]
        assert (dep[1:n] >= 1).all() and (dep[1:n] <= m_req[b]).all()
        assert all(0 <= par[x] < x for x in range(1, n))
        assert all(score[x] <= score[x - 1] for x in range(2, n))
        if n > 1:
            cut.append(score[n - 1])
    # everything taken scores at least as well as the best of what was left
    # of any request that still had room
    for b in range(B):
        n = int(t["n_nodes"][b])
        if n - 1 < N and drafts.sum() == budget and cut:
            ref = oracle.tree_build(tok[b:b + 1, : m_req[b]], sc[b:b + 1, : m_req[b]], root[b:b + 1], N)
            nxt = ref["node_score"][0, n] if n < N + 1 else -np.inf
            assert nxt <= min(cut)
