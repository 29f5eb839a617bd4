"""Pins for the oracle's argmax, acceptance and commit (CPU only).

What fixes the answer: torch.argmax (first-index rule), the hand-worked
acceptance cases in tests/golden, tau in [1, m+1], reduction of a chain tree
to plain speculative verification, the planted extremes (p = 1 accepts the
whole rank-0 chain present in the tree; an argmax outside the lattice accepts
nothing), exact KV-append copies, and multi-step consistency: after several
verify+commit steps the committed GDN state and KV cache equal a sequential
decode of the emitted token stream.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_best_gb300 import synth
from tests.indep import plain_chain_verify, root_path

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_argmax_matches_torch_first_index():
    g = torch.Generator().manual_seed(0)
    for dt in (torch.float32, torch.bfloat16):
        x = torch.randint(-3, 4, (64, 257), generator=g).to(dt)   # heavy ties
        idx, mar = oracle.argmax(x)
        np.testing.assert_array_equal(idx, torch.argmax(x.float(), dim=-1).numpy())
        srt = torch.sort(x.double(), dim=-1, descending=True).values
        np.testing.assert_array_equal(mar, (srt[:, 0] - srt[:, 1]).float().numpy())
        y = torch.randn(8, 151936, generator=g).to(dt)
        np.testing.assert_array_equal(oracle.argmax(y)[0], torch.argmax(y.float(), -1).numpy())


def test_hand_worked_acceptance():
    g = json.load(open(os.path.join(GOLD, "tree_hand_example.json")))
    tree = oracle.tree_build(np.array([g["lat_tok"]], np.int32),
                             np.array([g["lat_score"]], np.float32),
                             np.array([g["root_tok"]], np.int32), g["N"])
    for case in g["accept_cases"]:
        acc = oracle.accept(tree, np.array([case["argmax"]], np.int32), g["m"])
        tau = case["tau"]
        assert int(acc["accept_len"][0]) == tau, case["why"]
        assert acc["accept_nodes"][0, :tau].tolist() == case["path"]
        assert acc["out_tok"][0, :tau].tolist() == case["out_tok"]
        assert (acc["accept_nodes"][0, tau:] == -1).all() and (acc["out_tok"][0, tau:] == -1).all()
        assert int(acc["new_root"][0]) == case["out_tok"][-1]


def _planted(cfg, seed, p=None):
    g = torch.Generator().manual_seed(seed)
    tok, sc, root = synth.make_lattice(cfg, g)
    tree = oracle.tree_build(tok, sc, root, cfg.N)
    logits = synth.make_logits(cfg, g)
    synth.plant_logits(logits, tok, sc, tree["node_depth"], tree["n_nodes"],
                       cfg.p_plant if p is None else p, g)
    return tok, sc, tree, logits


@pytest.mark.parametrize("ci", [0, 1, 3])
def test_tau_in_range_and_path_valid(ci):
    cfg = synth.config(ci).replace(V=4096, B=min(synth.config(ci).B, 4))
    for seed in range(5):
        tok, sc, tree, logits = _planted(cfg, seed)
        am, _ = oracle.argmax(logits)
        acc = oracle.accept(tree, am, cfg.m)
        for b in range(cfg.B):
            tau = int(acc["accept_len"][b])
            assert 1 <= tau <= cfg.m + 1
            path = acc["accept_nodes"][b, :tau]
            assert path[0] == 0
            for a, c in zip(path[:-1], path[1:]):
                assert tree["node_parent"][b, c] == a
                assert tree["node_tok"][b, c] == am[b, a]          # lossless: equals argmax
            assert acc["out_tok"][b, tau - 1] == am[b, path[-1]]
            # the path stops because no child of the last node carries its argmax
            last = path[-1]
            kids = [c for c in range(int(tree["n_nodes"][b])) if tree["node_parent"][b, c] == last]
            assert all(tree["node_tok"][b, c] != am[b, last] for c in kids)


def test_chain_tree_is_plain_speculative_verification():
    cfg = synth.config(1).replace(K=1, N=8, V=64)
    for seed in range(30):
        tok, sc, tree, logits = _planted(cfg, seed, p=0.7)
        am, _ = oracle.argmax(logits)
        acc = oracle.accept(tree, am, cfg.m)
        drafts = tree["node_tok"][0, 1:].tolist()
        tau, out = plain_chain_verify(int(tree["node_tok"][0, 0]), drafts, am[0].tolist())
        assert int(acc["accept_len"][0]) == tau
        assert acc["out_tok"][0, :tau].tolist() == out


def test_p1_accepts_the_rank0_chain_in_the_tree():
    for ci in (0, 1, 2):
        cfg = synth.config(ci).replace(V=8192)
        for seed in range(3):
            tok, sc, tree, logits = _planted(cfg, seed, p=1.0)
            am, _ = oracle.argmax(logits)
            acc = oracle.accept(tree, am, cfg.m)
            # depth reached by following rank-0 children inside the tree
            d, cur = 0, 0
            while True:
                nxt = [c for c in range(int(tree["n_nodes"][0]))
                       if tree["node_parent"][0, c] == cur and tree["node_rank"][0, c] == 0]
                if not nxt:
                    break
                cur, d = nxt[0], d + 1
            assert int(acc["accept_len"][0]) == d + 1


def test_argmax_outside_lattice_accepts_nothing():
    cfg = synth.config(1).replace(V=8192)
    tok, sc, tree, logits = _planted(cfg, 0, p=0.0)
    first = set(tok[0, 0].tolist())
    outside = next(x for x in range(cfg.V) if x not in first)
    logits[0, 0, outside] = logits[0, 0].float().max() + 2
    am, _ = oracle.argmax(logits)
    acc = oracle.accept(tree, am, cfg.m)
    assert int(acc["accept_len"][0]) == 1
    assert acc["out_tok"][0, 0] == outside and acc["new_root"][0] == outside


def test_commit_kv_appends_accepted_rows():
    cfg = synth.config(0).replace(B=2)
    tok, sc, tree, logits = _planted(cfg, 3, p=0.9)
    acc = oracle.accept(tree, oracle.argmax(logits)[0], cfg.m)
    g = torch.Generator().manual_seed(9)
    lay = synth.make_attn_layer(cfg, g, Lmax=40)
    L = np.array([17, 30], np.int32)
    kc, vc = oracle.commit_kv(acc, lay["k_tree"], lay["v_tree"], lay["k_cache"], lay["v_cache"], L)
    for b in range(2):
        tau = int(acc["accept_len"][b])
        for s in range(tau):
            node = acc["accept_nodes"][b, s]
            np.testing.assert_array_equal(kc[b, L[b] + s], lay["k_tree"][b, node].numpy())
            np.testing.assert_array_equal(vc[b, L[b] + s], lay["v_tree"][b, node].numpy())
        untouched = [x for x in range(40) if not (L[b] <= x < L[b] + tau)]
        np.testing.assert_array_equal(kc[b, untouched], lay["k_cache"][b, untouched].numpy())
    with pytest.raises(ValueError):
        oracle.commit_kv(acc, lay["k_tree"], lay["v_tree"], lay["k_cache"], lay["v_cache"],
                         np.array([40, 0], np.int32))


def test_multi_step_state_equals_sequential_decode():
    """S verify+commit steps == a plain token-by-token decode of the stream."""
    cfg = synth.config(0).replace(B=2, Hk=2, Hv=4, dk=16, dv=8, Hq=4, Hkv=2, D=16, V=64)
    seed, steps, L0 = 11, 4, 5
    g = torch.Generator().manual_seed(seed)
    Lmax = L0 + steps * (cfg.m + 1)
    gdn = synth.make_gdn_layer(cfg, g)
    attn = synth.make_attn_layer(cfg, g, Lmax=Lmax)
    h = gdn["h0"].double().numpy().copy()
    h_init = h.copy()
    kc, vc = attn["k_cache"].numpy().copy(), attn["v_cache"].numpy().copy()
    kv_len = np.full(cfg.B, L0, np.int32)
    root = torch.randint(0, cfg.V, (cfg.B,), generator=g).int()
    stream = [[int(root[b])] for b in range(cfg.B)]      # tokens fed into the state
    taus = []
    for step in range(steps):
        gs = torch.Generator().manual_seed(1000 + step)
        tok, sc, _ = synth.make_lattice(cfg, gs)
        tree = oracle.tree_build(tok, sc, root, cfg.N)
        synth.fill_rows_by_token(cfg, seed, tree["node_tok"], tree["node_depth"],
                                 tree["n_nodes"], kv_len, [gdn], [attn])
        logits = synth.make_logits(cfg, gs)
        synth.plant_logits(logits, tok, sc, tree["node_depth"], tree["n_nodes"], 0.8, gs)
        acc = oracle.accept(tree, oracle.argmax(logits)[0], cfg.m)
        h = oracle.commit_gdn(acc, h, gdn["k"], gdn["v"], gdn["alpha"], gdn["beta"])
        kc, vc = oracle.commit_kv(acc, attn["k_tree"], attn["v_tree"], kc, vc, kv_len)
        kv_len = kv_len + acc["accept_len"]
        root = torch.as_tensor(acc["new_root"])
        for b in range(cfg.B):
            tau = int(acc["accept_len"][b])
            stream[b] += acc["out_tok"][b, :tau].tolist()
            taus.append(tau)
    assert max(taus) > 1                                  # some drafts were accepted

    for b in range(cfg.B):
        toks = stream[b][:-1]                             # the last bonus is still pending
        assert len(toks) == kv_len[b] - L0
        hb = h_init[b].copy()
        for pos, t in enumerate(toks, start=L0):
            gg = synth.row_generator(seed, 0, 0, b, pos, t)
            kq = torch.randn((2, cfg.Hk, cfg.dk), generator=gg)
            kq = kq / kq.norm(dim=-1, keepdim=True)
            k = kq[1].to(cfg.dtype).double().numpy()
            v = torch.randn((cfg.Hv, cfg.dv), generator=gg).to(cfg.dtype).double().numpy()
            be = torch.sigmoid(torch.randn((cfg.Hv,), generator=gg)).double().numpy()
            al = (0.9 + 0.1 * torch.rand((cfg.Hv,), generator=gg)).double().numpy()
            for j in range(cfg.Hv):
                kk = k[j // 2]
                hb[j] = al[j] * (np.eye(cfg.dk) - be[j] * np.outer(kk, kk)) @ hb[j] \
                    + be[j] * np.outer(kk, v[j])
            ga = synth.row_generator(seed, 1, 0, b, pos, t)
            torch.randn((cfg.Hq, cfg.D), generator=ga)    # attention q (not stored)
            kr = torch.randn((cfg.Hkv, cfg.D), generator=ga).to(cfg.dtype).numpy()
            vr = torch.randn((cfg.Hkv, cfg.D), generator=ga).to(cfg.dtype).numpy()
            np.testing.assert_array_equal(kc[b, pos], kr)
            np.testing.assert_array_equal(vc[b, pos], vr)
        err = np.linalg.norm(h[b] - hb) / np.linalg.norm(hb)
        assert err < 1e-12, err
