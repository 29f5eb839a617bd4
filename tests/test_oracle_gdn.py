"""Pins for the oracle's tree-masked Gated DeltaNet (CPU only).

What fixes the answer: a hand-worked two-row chain (tests/golden), closed
forms (beta = 0; zero state; the exact delta write), the head mapping, an
independent float64 ancestor-expansion formulation, and the defining property
that each node's output is the sequential chain decode of its own root path.
"""
import json
import os

import numpy as np
import torch

import oracle
from speculative_decoding_tree_best_gb300 import synth
from tests.indep import gdn_expand, root_path

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _chain_tree(T):
    par = np.arange(-1, T - 1, dtype=np.int32)[None]
    return dict(node_parent=par, n_nodes=np.array([T], np.int32))


def _tiny(seed=0, **kw):
    cfg = synth.config(0).replace(**kw)
    g = torch.Generator().manual_seed(seed)
    tok, sc, root = synth.make_lattice(cfg, g)
    tree = oracle.tree_build(tok, sc, root, cfg.N)
    lay = synth.make_gdn_layer(cfg, g)
    return cfg, tree, lay


def test_hand_worked_chain():
    g = json.load(open(os.path.join(GOLD, "gdn_hand_example.json")))
    rows = g["rows"]
    f = lambda key: np.array([[r[key]] for r in rows], np.float32)[None]   # [1][T][1][d]
    h0 = np.array(g["h0"], np.float64)[None, None]
    al = np.array([[[r["alpha"]] for r in rows]], np.float32)
    be = np.array([[[r["beta"]] for r in rows]], np.float32)
    o = oracle.gdn_tree(_chain_tree(2), h0, f("q"), f("k"), f("v"), al, be)
    np.testing.assert_array_equal(o[0, :, 0, :], np.array(g["expect_o"]))
    acc = dict(accept_len=np.array([1], np.int32), accept_nodes=np.array([[0, -1]], np.int32))
    h1 = oracle.commit_gdn(acc, h0, f("k"), f("v"), al, be)
    np.testing.assert_array_equal(h1[0, 0], np.array(g["expect_h_after_root"]))
    acc2 = dict(accept_len=np.array([2], np.int32), accept_nodes=np.array([[0, 1]], np.int32))
    h2 = oracle.commit_gdn(acc2, h0, f("k"), f("v"), al, be)
    np.testing.assert_array_equal(h2[0, 0], np.array(g["expect_h_after_child"]))


def test_beta_zero_is_pure_decay():
    cfg, tree, lay = _tiny(1)
    lay["beta"].zero_()
    o = oracle.gdn_tree(tree, lay["h0"], lay["q"], lay["k"], lay["v"], lay["alpha"], lay["beta"])
    par = tree["node_parent"][0]
    al = lay["alpha"][0].double().numpy()
    h0 = lay["h0"][0].double().numpy()
    q = lay["q"][0].double().numpy()
    for n in range(int(tree["n_nodes"][0])):
        A = np.prod(al[root_path(par, n)], axis=0)            # [Hv]
        for j in range(cfg.Hv):
            want = A[j] * (h0[j].T @ q[n, j * cfg.Hk // cfg.Hv])
            np.testing.assert_allclose(o[0, n, j], want, rtol=1e-12, atol=1e-15)


def test_zero_state_single_root():
    cfg = synth.config(0).replace(Hk=2, Hv=4)
    g = torch.Generator().manual_seed(2)
    lay = synth.make_gdn_layer(cfg, g, rows=1)
    lay["h0"].zero_()
    o = oracle.gdn_tree(_chain_tree(1), lay["h0"], lay["q"], lay["k"], lay["v"],
                        lay["alpha"], lay["beta"])
    q, k, v = (lay[x][0, 0].double().numpy() for x in ("q", "k", "v"))
    be = lay["beta"][0, 0].double().numpy()
    for j in range(4):
        i = j // 2                                              # repeat-interleave head map
        np.testing.assert_allclose(o[0, 0, j], be[j] * (k[i] @ q[i]) * v[j], rtol=1e-13)


def test_exact_delta_write():
    # alpha = beta = 1 and a unit basis key: the write replaces the value
    # stored under k, so reading it back with q = k returns v exactly.
    rng = np.random.default_rng(3)
    dk = dv = 8
    h0 = rng.normal(size=(1, 1, dk, dv))
    k = np.zeros((1, 1, 1, dk), np.float32)
    k[..., 3] = 1.0
    v = rng.normal(size=(1, 1, 1, dv)).astype(np.float32)
    one = np.ones((1, 1, 1), np.float32)
    o = oracle.gdn_tree(_chain_tree(1), h0, k, k, v, one, one)
    np.testing.assert_array_equal(o[0, 0, 0], v[0, 0, 0].astype(np.float64))


def test_matches_ancestor_expansion():
    for seed in range(4):
        cfg, tree, lay = _tiny(seed, Hk=2, Hv=4)
        o = oracle.gdn_tree(tree, lay["h0"], lay["q"], lay["k"], lay["v"], lay["alpha"],
                            lay["beta"])
        n = int(tree["n_nodes"][0])
        want, _ = gdn_expand(tree["node_parent"][0], n, lay["h0"][0], lay["q"][0], lay["k"][0],
                             lay["v"][0], lay["alpha"][0], lay["beta"][0])
        err = np.linalg.norm(o[0, :n] - want[:n]) / np.linalg.norm(want[:n])
        assert err < 1e-12, err
        assert not o[0, n:].any()


def test_bf16_inputs_match_ancestor_expansion():
    cfg = synth.config(1).replace(N=12, m=4, K=4, V=1000, Hk=2, Hv=4, dk=32, dv=16)
    g = torch.Generator().manual_seed(5)
    tok, sc, root = synth.make_lattice(cfg, g)
    tree = oracle.tree_build(tok, sc, root, cfg.N)
    lay = synth.make_gdn_layer(cfg, g)
    assert lay["q"].dtype == torch.bfloat16
    o = oracle.gdn_tree(tree, lay["h0"], lay["q"], lay["k"], lay["v"], lay["alpha"], lay["beta"])
    want, _ = gdn_expand(tree["node_parent"][0], cfg.T, lay["h0"][0], lay["q"][0].float(),
                         lay["k"][0].float(), lay["v"][0].float(), lay["alpha"][0], lay["beta"][0])
    assert np.linalg.norm(o[0] - want) / np.linalg.norm(want) < 1e-12


def test_each_node_equals_chain_decode_of_its_root_path():
    cfg, tree, lay = _tiny(6)
    o = oracle.gdn_tree(tree, lay["h0"], lay["q"], lay["k"], lay["v"], lay["alpha"], lay["beta"])
    par = tree["node_parent"][0]
    for n in range(int(tree["n_nodes"][0])):
        path = root_path(par, n)
        sub = {x: lay[x][:, path].contiguous() for x in ("q", "k", "v", "alpha", "beta")}
        oc = oracle.gdn_tree(_chain_tree(len(path)), lay["h0"], sub["q"], sub["k"], sub["v"],
                             sub["alpha"], sub["beta"])
        np.testing.assert_array_equal(o[0, n], oc[0, -1])


def test_commit_state_is_state_at_last_accepted_node():
    cfg, tree, lay = _tiny(7, Hk=2, Hv=4)
    n_nodes = int(tree["n_nodes"][0])
    _, states = gdn_expand(tree["node_parent"][0], n_nodes, lay["h0"][0], lay["q"][0],
                           lay["k"][0], lay["v"][0], lay["alpha"][0], lay["beta"][0])
    for last in range(n_nodes):
        path = root_path(tree["node_parent"][0], last)
        nodes = np.full((1, cfg.m + 1), -1, np.int32)
        nodes[0, :len(path)] = path
        acc = dict(accept_len=np.array([len(path)], np.int32), accept_nodes=nodes)
        h = oracle.commit_gdn(acc, lay["h0"], lay["k"], lay["v"], lay["alpha"], lay["beta"])
        err = np.linalg.norm(h[0] - states[last]) / np.linalg.norm(states[last])
        assert err < 1e-12, (last, err)
