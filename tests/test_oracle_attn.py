"""Pins for the oracle's tree-ancestor-masked attention (CPU only).

What fixes the answer: a hand-worked two-row example (tests/golden), float64
scaled_dot_product_attention (a library routine) on a chain tree with a causal
mask, and on every node of a bushy tree with its visible set gathered
explicitly, q = 0 giving the mean of the visible values, a single visible key
returning its value, and the GQA head mapping.
"""
import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from speculative_decoding_tree_best_gb300 import synth
from tests.indep import root_path

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _tree_from_parent(parent):
    T = len(parent)
    anc = np.zeros((1, T, 2), np.uint64)
    for n in range(T):
        for a in root_path(parent, n):
            anc[0, n, a // 64] |= np.uint64(1) << np.uint64(a % 64)
    return dict(node_parent=np.array([parent], np.int32), n_nodes=np.array([T], np.int32),
                node_anc=anc)


def _tiny(seed, **kw):
    cfg = synth.config(0).replace(**kw)
    g = torch.Generator().manual_seed(seed)
    tok, sc, root = synth.make_lattice(cfg, g)
    tree = oracle.tree_build(tok, sc, root, cfg.N)
    lay = synth.make_attn_layer(cfg, g)
    return cfg, tree, lay


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLD, "attn_hand_example.json")))
    ln3 = math.log(3.0)
    fix = lambda rows: np.array([[ln3 if x == "ln3" else x for x in r] for r in rows], np.float32)
    kt, vt, q = fix(g["k_tree"])[None, :, None], fix(g["v_tree"])[None, :, None], fix(g["q"])[None, :, None]
    kc, vc = fix(g["k_cache"])[None, :, None], fix(g["v_cache"])[None, :, None]
    o = oracle.attn_tree(_tree_from_parent(g["node_parent"]), q, kt, vt, kc, vc,
                         np.array([g["kv_len"]], np.int32))
    np.testing.assert_allclose(o[0, :, 0], np.array(g["expect_o"]), rtol=1e-6, atol=1e-6)


def test_chain_matches_causal_sdpa():
    cfg = synth.config(0).replace(Hq=4, Hkv=2)
    g = torch.Generator().manual_seed(1)
    T, L = 6, 37
    lay = synth.make_attn_layer(cfg, g, rows=T, Lmax=L + 5)
    tree = _tree_from_parent(list(range(-1, T - 1)))
    o = oracle.attn_tree(tree, lay["q"], lay["k_tree"], lay["v_tree"], lay["k_cache"],
                         lay["v_cache"], np.array([L], np.int32))
    k = torch.cat([lay["k_cache"][0, :L], lay["k_tree"][0]], 0).double()      # [L+T][Hkv][D]
    v = torch.cat([lay["v_cache"][0, :L], lay["v_tree"][0]], 0).double()
    q = lay["q"][0].double()                                                  # [T][Hq][D]
    k = k.repeat_interleave(2, dim=1).transpose(0, 1)                         # [Hq][L+T][D]
    v = v.repeat_interleave(2, dim=1).transpose(0, 1)
    mask = torch.ones(T, L + T, dtype=torch.bool)
    mask[:, L:] = torch.tril(torch.ones(T, T, dtype=torch.bool))
    want = F.scaled_dot_product_attention(q.transpose(0, 1), k, v, attn_mask=mask)
    np.testing.assert_allclose(o[0], want.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)


def test_every_node_matches_sdpa_over_its_visible_set():
    for seed in range(3):
        cfg, tree, lay = _tiny(seed, Hq=4, Hkv=2)
        L = 50 + seed
        o = oracle.attn_tree(tree, lay["q"], lay["k_tree"], lay["v_tree"], lay["k_cache"],
                             lay["v_cache"], np.array([L], np.int32))
        par = tree["node_parent"][0]
        for n in range(int(tree["n_nodes"][0])):
            path = root_path(par, n)
            k = torch.cat([lay["k_cache"][0, :L], lay["k_tree"][0, path]], 0).double()
            v = torch.cat([lay["v_cache"][0, :L], lay["v_tree"][0, path]], 0).double()
            for h in range(cfg.Hq):
                want = F.scaled_dot_product_attention(
                    lay["q"][0, n, h].double()[None, None], k[:, h // 2][None], v[:, h // 2][None])
                np.testing.assert_allclose(o[0, n, h], want[0, 0].numpy(), rtol=1e-10, atol=1e-12)


def test_zero_query_is_mean_of_visible_values():
    cfg, tree, lay = _tiny(4, Hq=4, Hkv=2)
    lay["q"].zero_()
    L = 20
    o = oracle.attn_tree(tree, lay["q"], lay["k_tree"], lay["v_tree"], lay["k_cache"],
                         lay["v_cache"], np.array([L], np.int32))
    par = tree["node_parent"][0]
    for n in range(int(tree["n_nodes"][0])):
        vis = torch.cat([lay["v_cache"][0, :L], lay["v_tree"][0, root_path(par, n)]], 0).double()
        for h in range(cfg.Hq):
            np.testing.assert_allclose(o[0, n, h], vis[:, h // 2].mean(0).numpy(), rtol=1e-12)


def test_single_visible_key_returns_its_value():
    cfg, tree, lay = _tiny(5)
    o = oracle.attn_tree(tree, lay["q"], lay["k_tree"], lay["v_tree"], lay["k_cache"],
                         lay["v_cache"], np.array([0], np.int32))
    np.testing.assert_allclose(o[0, 0], lay["v_tree"][0, 0].double().numpy(), rtol=1e-12)


def test_padding_rows_are_zero():
    cfg = synth.config(0).replace(m=1, K=2, N=6)
    g = torch.Generator().manual_seed(6)
    tok, sc, root = synth.make_lattice(cfg, g)
    tree = oracle.tree_build(tok, sc, root, cfg.N)
    assert int(tree["n_nodes"][0]) == 3
    lay = synth.make_attn_layer(cfg, g)
    o = oracle.attn_tree(tree, lay["q"], lay["k_tree"], lay["v_tree"], lay["k_cache"],
                         lay["v_cache"], np.array([10], np.int32))
    assert not o[0, 3:].any() and o[0, :3].any()
