"""Pins for the oracle's Markov-head edge scores and the tree built on them
(CPU only).

DSpark's Markov head (digest, prerequisites / parallel drafter) scores a
candidate y after the previous token x as l(y) = bases(y) + <W1[x], W2[y]>;
with edges scored log p(child | parent) (technical novelty), a child's edge is
l minus the log-sum-exp over the position's candidates under that parent.

What fixes the answer: the fp32 exp/log against libm's error bounds, the edge
scores against a float64 evaluation, the exact reduction to the plain tree
when W1 = W2 = 0, and brute force over tiny lattices with parent-dependent
ranks.
"""
import numpy as np
import pytest

import oracle
from tests.indep import brute_force_markov


def test_exp32_log32_error_bounds():
    x = -np.concatenate([np.linspace(0, 86, 40001), np.geomspace(1e-8, 1, 2001)]).astype(np.float32)
    z = np.concatenate([np.linspace(1, 64, 40001), 1 + np.geomspace(1e-7, 1, 2001)]).astype(np.float32)
    ex, lz = oracle.exp32_log32(x, z)
    e64 = np.exp(x.astype(np.float64))
    assert (np.abs(ex - e64) / e64).max() < 2 * 2.0 ** -23          # within 2 ulp
    l64 = np.log(z.astype(np.float64))
    assert np.abs(lz - l64).max() < 5e-7                          # ~1 ulp of log(64)
    assert ex[x == 0].tolist() == [1.0] * int((x == 0).sum()) and lz[z == 1].tolist() == [0.0] * int((z == 1).sum())


def _markov(rng, m, K, V=64, R=8, zero=False):
    tok = np.stack([rng.permutation(V)[:K] for _ in range(m)]).astype(np.int32)
    base = (rng.normal(0, 2, size=(m, K))).astype(np.float32)
    sd = R ** -0.25
    W1 = (rng.normal(0, sd, size=(V, R))).astype(np.float32)
    W2 = (rng.normal(0, sd, size=(V, R))).astype(np.float32)
    if zero:
        W1[:] = 0
        W2[:] = 0
    return tok, base, W1, W2


def test_edges_against_float64():
    rng = np.random.default_rng(11)
    for _ in range(200):
        K = int(rng.integers(1, 17))
        tok, base, W1, W2 = _markov(rng, 1, K, R=32)
        x = int(rng.integers(0, 64))
        e = oracle.markov_edges(x, tok[0], base[0], W1, W2)
        l64 = base[0].astype(np.float64) + W2[tok[0]].astype(np.float64) @ W1[x].astype(np.float64)
        m = l64.max()
        want = l64 - (m + np.log(np.exp(l64 - m).sum()))
        assert np.abs(e - want).max() < 2e-5
        assert abs(np.log(np.exp(e.astype(np.float64)).sum())) < 1e-5   # a distribution


def test_zero_markov_term_is_the_plain_tree():
    rng = np.random.default_rng(12)
    for _ in range(50):
        m, K = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        N = int(rng.integers(0, 40))
        tok, base, W1, W2 = _markov(rng, m, K, zero=True)
        root = np.array([int(rng.integers(0, 64))], np.int32)
        # with W = 0 the edges do not depend on the parent: the plain tree over them
        sc = np.stack([oracle.markov_edges(0, tok[d], base[d], W1, W2) for d in range(m)])
        t = oracle.tree_build_markov(tok[None], base[None], W1, W2, root, N)
        ref = oracle.tree_build(tok[None], sc[None], root, N)
        for k in ref:
            if k == "node_score":
                np.testing.assert_array_equal(t[k].view(np.uint32), ref[k].view(np.uint32))
            else:
                np.testing.assert_array_equal(t[k], ref[k], err_msg=k)


@pytest.mark.parametrize("R", [4, 16])
def test_markov_tree_equals_brute_force(R):
    rng = np.random.default_rng(13 + R)
    differs = 0
    for trial in range(150):
        m, K = int(rng.integers(1, 4)), int(rng.integers(1, 5))
        total = sum(K ** d for d in range(1, m + 1))
        N = int(rng.integers(0, total + 3))
        tok, base, W1, W2 = _markov(rng, m, K, R=R)
        root = int(rng.integers(0, 64))
        t = oracle.tree_build_markov(tok[None], base[None], W1, W2, np.array([root], np.int32), N)
        bf = brute_force_markov(tok, base, W1, W2, root, N,
                                lambda x, d: oracle.markov_edges(x, tok[d], base[d], W1, W2))
        assert int(t["n_nodes"][0]) == bf["n_nodes"] == 1 + min(N, total)
        for k in ("node_tok", "node_parent", "node_depth", "node_rank", "node_anc"):
            np.testing.assert_array_equal(t[k][0], bf[k], err_msg=f"{k} trial {trial}")
        np.testing.assert_array_equal(t["node_score"][0].view(np.uint32),
                                      bf["node_score"].view(np.uint32))
        # the Markov term changes some trees (the ranks depend on the parent)
        z = oracle.tree_build_markov(tok[None], base[None], 0 * W1, 0 * W2,
                                     np.array([root], np.int32), N)
        differs += int(not np.array_equal(z["node_tok"], t["node_tok"]))
    assert differs > 10
