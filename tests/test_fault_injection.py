"""Host-side fault injection: the parity harness must reject a system with an
injected fault and accept a correct one.

The SpecPilot digest (prerequisites: reward hacking and token forcing) rejects
systems that gain speed through a numerical shortcut such as a logit bias on
part of the vocabulary.  Here the "system under test" is the CPU oracle run on
perturbed inputs (or with a perturbed output), packaged like a GPU step; the
harness compares it with the oracle on the clean inputs.  No GPU is used."""
import types

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_best_gb300 import synth
from tests import parity


class _Tree:
    def __init__(self, t):
        self._t = t

    def to_numpy(self):
        return self._t


def _oracle_system(scfg, inp):
    """One full oracle step on `inp`, packaged with the attributes the harness
    reads from a GPU step."""
    tree = oracle.tree_build(inp["lat_tok"], inp["lat_score"], inp["root_tok"], scfg.N)
    gdn_o = torch.stack([torch.from_numpy(oracle.gdn_tree(tree, l["h0"], l["q"], l["k"], l["v"],
                                                          l["alpha"], l["beta"]))
                         for l in inp["gdn"]])
    attn_o = torch.stack([torch.from_numpy(oracle.attn_tree(tree, l["q"], l["k_tree"],
                                                            l["v_tree"], l["k_cache"],
                                                            l["v_cache"], inp["kv_len"]))
                          for l in inp["attn"]])
    am, _ = oracle.argmax(inp["logits"])
    acc = oracle.accept(tree, am, scfg.m)
    h0 = torch.stack([torch.from_numpy(oracle.commit_gdn(acc, l["h0"], l["k"], l["v"],
                                                         l["alpha"], l["beta"]))
                      for l in inp["gdn"]])
    kc, vc = [], []
    for l in inp["attn"]:
        k, v = oracle.commit_kv(acc, l["k_tree"], l["v_tree"], l["k_cache"], l["v_cache"],
                                inp["kv_len"])
        kc.append(torch.from_numpy(np.asarray(k)))
        vc.append(torch.from_numpy(np.asarray(v)))
    L0 = inp["kv_len"].numpy()
    ok = L0 + acc["accept_len"] <= scfg.Lmax
    x = {"kv_len": torch.from_numpy(np.where(ok, L0 + acc["accept_len"], L0).astype(np.int32)),
         "root_tok": torch.from_numpy(np.where(ok, acc["new_root"],
                                               inp["root_tok"].numpy()).astype(np.int32)),
         "gdn_h0": h0, "k_cache": torch.stack(kc), "v_cache": torch.stack(vc)}
    accs = types.SimpleNamespace(argmax=torch.from_numpy(np.asarray(am)),
                                 **{k: torch.from_numpy(np.asarray(acc[k]))
                                    for k in ("accept_len", "accept_nodes", "out_tok")})
    return types.SimpleNamespace(tree=_Tree(tree), gdn_o=gdn_o, attn_o=attn_o, acc=accs, x=x)


@pytest.fixture(scope="module")
def clean():
    scfg = synth.config(0)
    inp, tree = parity.prepare(scfg, 3)
    return scfg, inp, tree


def _clone(inp):
    out = {}
    for k, v in inp.items():
        if isinstance(v, torch.Tensor):
            out[k] = v.clone()
        elif isinstance(v, list):
            out[k] = [{kk: vv.clone() for kk, vv in lay.items()} for lay in v]
        else:
            out[k] = v
    return out


def test_harness_accepts_the_correct_system(clean):
    scfg, inp, tree = clean
    sut = _oracle_system(scfg, _clone(inp))
    r = parity.compare(scfg, inp, tree, sut)
    assert r["gdn_rel_l2"] < 1e-6 and r["attn_rel_l2"] < 1e-6     # fp32 read-back only


def test_logit_bias_on_part_of_the_vocabulary_is_rejected(clean):
    scfg, inp, tree = clean
    bad = _clone(inp)
    favoured = torch.randperm(scfg.V, generator=torch.Generator().manual_seed(1))[:64]
    bad["logits"][:, :, favoured] += 5.0
    sut = _oracle_system(scfg, bad)
    with pytest.raises(AssertionError):
        parity.compare(scfg, inp, tree, sut)


def test_flipped_lattice_score_is_rejected(clean):
    scfg, inp, tree = clean
    bad = _clone(inp)
    s0 = bad["lat_score"][0, 0]
    s0[torch.argmax(s0)] = -50.0          # the best first-position candidate drops out
    sut = _oracle_system(scfg, bad)
    with pytest.raises(AssertionError):
        parity.compare(scfg, inp, tree, sut)


def test_lossy_gdn_shortcut_is_rejected(clean):
    scfg, inp, tree = clean
    sut = _oracle_system(scfg, _clone(inp))
    sut.gdn_o[:, :, :, 0] *= 1.01         # one head 1% off: rel-L2 ~5e-3
    with pytest.raises(AssertionError, match="GDN"):
        parity.compare(scfg, inp, tree, sut)


def _bigger():
    """A case with enough rows that one bad row hides in the whole-tensor
    figure: 2 requests, N = 20, 8 v-heads / 8 q-heads."""
    scfg = synth.config(0).replace(B=2, m=4, K=4, N=20, Hk=4, Hv=8, Hq=8, Hkv=2, L=64, V=256)
    inp, tree = parity.prepare(scfg, 5)
    return scfg, inp, tree


@pytest.mark.parametrize("what", ["gdn", "attn", "state"])
def test_one_bad_row_is_caught_by_the_row_bound(what):
    """A 2% error on a single (request, node, head) row -- or on one row of one
    committed state -- stays under the whole-tensor 2e-3 bound but breaks the
    per-row bound."""
    scfg, inp, tree = _bigger()
    sut = _oracle_system(scfg, _clone(inp))
    if what == "gdn":
        sut.gdn_o[0, 1, 7, 3] *= 1.02                      # request 1, node 7, v-head 3
        t = sut.gdn_o[0]
    elif what == "attn":
        sut.attn_o[0, 0, 12, 5] *= 1.02                    # request 0, node 12, q-head 5
        t = sut.attn_o[0]
    else:
        sut.x["gdn_h0"][0, 1, 2, 17] *= 1.02               # request 1, v-head 2, d_k row 17
        t = sut.x["gdn_h0"][0]
    assert float(t.double().norm()) > 0
    with pytest.raises(AssertionError, match="row"):
        parity.compare(scfg, inp, tree, sut)
    # the whole-tensor figure alone would have let it through
    clean_sut = _oracle_system(scfg, _clone(inp))
    ref = {"gdn": clean_sut.gdn_o[0], "attn": clean_sut.attn_o[0],
           "state": clean_sut.x["gdn_h0"][0]}[what]
    assert parity.rel_l2(t.double().numpy(), ref.double().numpy()) < parity.REL_L2
