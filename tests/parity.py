"""Parity harness: run one verify step through the CUDA library and the same
step through the CPU oracle on identical seeded inputs, and compare.

Contract (the tree-verify library's parity bar):
  * bit-exact: tree topology/scores, argmax -- or, at temperature > 0, each
    row's draw -- (except rows whose top-2 margin is below 1e-3, where the
    GPU's token must be within 1e-3 of the best and the walk is checked on the
    GPU's token), accepted lengths/paths, emitted tokens, KV-cache rows,
    kv_len and the new root token;
  * rel-L2 <= 2e-3 (computed in float64 against the float64 oracle) for GDN
    outputs, attention outputs and committed GDN states, over each layer's
    whole tensor; and rel-L2 <= 6e-3 on every single row: each (request,
    node, head) output row and each row of each committed (request, head)
    state.  bf16 rounding of the outputs alone contributes about 1.65e-3 to a
    whole tensor and up to ~2.2e-3 to one 128-element row, so the GPU must keep
    everything else in fp32; the row bound catches an error confined to one
    node, depth or head, which the whole-tensor figure would average away.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decoding_tree_best_gb300 import synth
from speculative_decoding_tree_best_gb300.step import VerifyStep, stack_inputs

REL_L2 = 2e-3
ROW_REL_L2 = 6e-3
MARGIN_EXEMPT = 1e-3


def rel_l2(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    num = np.linalg.norm(got - want)
    return float(num / den) if den > 0 else float(num)


def row_rel_l2(got, want, valid=None):
    """Worst rel-L2 over the rows of the last axis: (error, index of that row
    in the leading axes).  valid: boolean mask over the leading axes (rows
    outside it are not compared)."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    num = np.linalg.norm(got - want, axis=-1)
    den = np.linalg.norm(want, axis=-1)
    err = np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
    if valid is not None:
        err = np.where(valid, err, 0.0)
    i = int(np.argmax(err))
    return float(err.reshape(-1)[i]), np.unravel_index(i, err.shape)


def _node_rows(nn, req, T, heads):
    """[len(req)][T][heads] mask of the real tree rows of each request."""
    v = np.zeros((len(req), T, heads), bool)
    for i, b in enumerate(req):
        v[i, :nn[b]] = True
    return v


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def prepare(scfg: synth.SpecConfig, seed: int, kv_len=None, lat_edit=None):
    """CPU inputs with logits planted from the oracle's tree."""
    inp = synth.make_step_inputs(scfg, seed)
    if kv_len is not None:
        inp["kv_len"] = torch.as_tensor(kv_len, dtype=torch.int32).reshape(scfg.B)
    if lat_edit is not None:
        lat_edit(inp)
    if scfg.markov_R > 0:
        tree = oracle.tree_build_markov(inp["lat_tok"], inp["lat_base"], inp["W1"], inp["W2"],
                                        inp["root_tok"], scfg.N)
    elif scfg.ragged:
        tree = oracle.tree_build_ragged(inp["lat_tok"], inp["lat_score"], inp["root_tok"], scfg.N,
                                        inp["m_req"], scfg.budget)
    else:
        tree = oracle.tree_build(inp["lat_tok"], inp["lat_score"], inp["root_tok"], scfg.N)
    fc = (synth.first_child_tokens(tree["node_parent"], tree["node_rank"], tree["node_tok"],
                                   tree["n_nodes"]) if scfg.markov_R > 0 else None)
    synth.plant_logits(inp["logits"], inp["lat_tok"], inp["lat_score"], tree["node_depth"],
                       tree["n_nodes"], scfg.p_plant, inp["plant_gen"], first_child=fc,
                       gap=scfg.plant_gap)
    return inp, tree


def run_gpu(scfg, inp, calls=False, persistent=False):
    """One step on the GPU: one spec_verify_step call (the persistent variant
    with persistent=True), or (calls=True) the four single-operation calls."""
    x = stack_inputs(inp, "cuda")
    st = VerifyStep(scfg, x, persistent=persistent)
    if calls:
        st.run_calls()
    else:
        st.run()
    torch.cuda.synchronize()
    return st


def compare(scfg, inp, tree_o, st, req=None, attn_kv_heads=None, gdn_layers=None,
            attn_layers=None) -> dict:
    """Compare every output of one GPU step with the oracle.

    req: request indices the float checks sample (all when None);
    attn_kv_heads: kv-heads the attention check samples (all when None).
    Returns a dict of measured errors; raises AssertionError on any breach.
    """
    B, T, m = scfg.B, scfg.T, scfg.m
    req = list(range(B)) if req is None else list(req)
    res = {}

    # ---- tree: bit-exact -------------------------------------------------------
    tg = st.tree.to_numpy()
    for k in ("node_tok", "node_parent", "node_depth", "node_rank", "n_nodes"):
        np.testing.assert_array_equal(tg[k], tree_o[k], err_msg=k)
    np.testing.assert_array_equal(tg["node_score"].view(np.uint32),
                                  tree_o["node_score"].view(np.uint32), err_msg="node_score bits")
    np.testing.assert_array_equal(tg["node_anc"], tree_o["node_anc"], err_msg="node_anc")
    nn = tree_o["n_nodes"]

    # ---- GDN outputs ----------------------------------------------------------------
    gl = range(scfg.n_gdn) if gdn_layers is None else gdn_layers
    worst = worst_row = 0.0
    for l in gl:
        lay = inp["gdn"][l]
        sub = {k: lay[k][req] for k in ("h0", "q", "k", "v", "alpha", "beta")}
        tsub = {k: tree_o[k][req] for k in ("node_parent", "n_nodes")}
        want = oracle.gdn_tree(tsub, sub["h0"], sub["q"], sub["k"], sub["v"], sub["alpha"],
                               sub["beta"])
        got = _f64(st.gdn_o[l][req])
        for i, b in enumerate(req):
            assert not got[i, nn[b]:].any(), "GDN padding rows must be zero"
        e = rel_l2(got, want)
        assert e <= REL_L2, f"GDN layer {l}: rel-L2 {e:.3e}"
        worst = max(worst, e)
        er, at = row_rel_l2(got, want, _node_rows(nn, req, T, got.shape[2]))
        assert er <= ROW_REL_L2, \
            f"GDN layer {l}: row (request {req[at[0]]}, node {at[1]}, v-head {at[2]}) rel-L2 {er:.3e}"
        worst_row = max(worst_row, er)
    res["gdn_rel_l2"] = worst
    res["gdn_row_rel_l2"] = worst_row

    # ---- attention outputs --------------------------------------------------------
    al = range(scfg.n_attn) if attn_layers is None else attn_layers
    G = scfg.Hq // scfg.Hkv
    kvh = list(range(scfg.Hkv)) if attn_kv_heads is None else list(attn_kv_heads)
    qh = [g * G + i for g in kvh for i in range(G)]
    worst = worst_row = 0.0
    kv_len = inp["kv_len"]              # read-only input of the step (restored below)
    for l in al:
        lay = inp["attn"][l]
        want = oracle.attn_tree(
            {k: tree_o[k][req] for k in ("n_nodes", "node_anc")},
            lay["q"][req][:, :, qh].contiguous(), lay["k_tree"][req][:, :, kvh].contiguous(),
            lay["v_tree"][req][:, :, kvh].contiguous(), lay["k_cache"][req][:, :, kvh].contiguous(),
            lay["v_cache"][req][:, :, kvh].contiguous(), kv_len[req])
        got = _f64(st.attn_o[l][req][:, :, qh])
        for i, b in enumerate(req):
            assert not got[i, nn[b]:].any(), "attention padding rows must be zero"
        e = rel_l2(got, want)
        assert e <= REL_L2, f"attention layer {l}: rel-L2 {e:.3e}"
        worst = max(worst, e)
        er, at = row_rel_l2(got, want, _node_rows(nn, req, T, got.shape[2]))
        assert er <= ROW_REL_L2, (f"attention layer {l}: row (request {req[at[0]]}, node {at[1]}, "
                                  f"q-head {qh[at[2]]}) rel-L2 {er:.3e}")
        worst_row = max(worst_row, er)
    res["attn_rel_l2"] = worst
    res["attn_row_rel_l2"] = worst_row

    # ---- argmax (or draw) + acceptance: bit-exact -------------------------------------
    kv_len = inp["kv_len"]
    sampled = scfg.temperature > 0
    if sampled:
        am_o, margin = oracle.sample_rows(inp["logits"], nn, kv_len, scfg.temperature,
                                          scfg.sample_seed)
    else:
        am_o, margin = oracle.argmax(inp["logits"])
    am_g = st.acc.argmax.cpu().numpy()
    rows = am_o.copy()
    exempt = 0
    for b in range(B):
        for t in range(T):
            if t >= nn[b]:
                assert am_g[b, t] == -1
            elif am_g[b, t] != am_o[b, t]:
                what = "draw" if sampled else "argmax"
                assert margin[b, t] < MARGIN_EXEMPT, f"{what} row ({b},{t})"
                g = int(am_g[b, t])
                assert 0 <= g < scfg.V, f"{what} row ({b},{t}) out of range"
                if sampled:                       # the GPU's token nearly ties the draw
                    gaps = oracle.sample_gaps(inp["logits"][b, t], t, b, int(kv_len[b]),
                                              scfg.temperature, scfg.sample_seed, g)
                    assert max(gaps) < MARGIN_EXEMPT, f"draw row ({b},{t}) gaps {gaps}"
                else:
                    row = inp["logits"][b, t].float()
                    assert float(row[g]) >= float(row.max()) - MARGIN_EXEMPT
                rows[b, t] = g                    # check the walk on the GPU's token
                exempt += 1
    res["exempt_rows"] = exempt
    acc_o = oracle.accept(tree_o, rows, m)
    np.testing.assert_array_equal(st.acc.accept_len.cpu().numpy(), acc_o["accept_len"])
    np.testing.assert_array_equal(st.acc.accept_nodes.cpu().numpy(), acc_o["accept_nodes"])
    np.testing.assert_array_equal(st.acc.out_tok.cpu().numpy(), acc_o["out_tok"])
    res["tau"] = acc_o["accept_len"].tolist()

    # ---- commit ------------------------------------------------------------------------
    L0 = kv_len.numpy()
    ok = L0 + acc_o["accept_len"] <= scfg.Lmax
    new_len = np.where(ok, L0 + acc_o["accept_len"], L0)
    np.testing.assert_array_equal(st.x["kv_len"].cpu().numpy(), new_len)
    np.testing.assert_array_equal(st.x["root_tok"].cpu().numpy(),
                                  np.where(ok, acc_o["new_root"], inp["root_tok"].numpy()))
    worst = worst_row = 0.0
    for l in gl:
        lay = inp["gdn"][l]
        acc_r = {k: acc_o[k][req] for k in ("accept_len", "accept_nodes")}
        want = oracle.commit_gdn(acc_r, lay["h0"][req], lay["k"][req], lay["v"][req],
                                 lay["alpha"][req], lay["beta"][req])
        got = _f64(st.x["gdn_h0"][l][req])
        for i, b in enumerate(req):
            if not ok[b]:
                np.testing.assert_array_equal(got[i], lay["h0"][b].double().numpy())
                continue
            e = rel_l2(got[i], want[i])
            assert e <= REL_L2, f"committed state layer {l} request {b}: rel-L2 {e:.3e}"
            worst = max(worst, e)
            er, at = row_rel_l2(got[i], want[i])
            assert er <= ROW_REL_L2, (f"committed state layer {l} request {b}: row (v-head "
                                      f"{at[0]}, d_k row {at[1]}) rel-L2 {er:.3e}")
            worst_row = max(worst_row, er)
    res["state_rel_l2"] = worst
    res["state_row_rel_l2"] = worst_row
    for l in al:
        lay = inp["attn"][l]
        kc_g = st.x["k_cache"][l][req].cpu()
        vc_g = st.x["v_cache"][l][req].cpu()
        for i, b in enumerate(req):
            kc_w, vc_w = lay["k_cache"][b].clone(), lay["v_cache"][b].clone()
            if ok[b]:
                tau = int(acc_o["accept_len"][b])
                for s in range(tau):
                    node = int(acc_o["accept_nodes"][b, s])
                    kc_w[L0[b] + s] = lay["k_tree"][b, node]
                    vc_w[L0[b] + s] = lay["v_tree"][b, node]
            assert torch.equal(kc_g[i], kc_w) and torch.equal(vc_g[i], vc_w), \
                f"KV cache layer {l} request {b}"
    res["overflow"] = (~ok).tolist()
    return res


def check_case(scfg, seed, **kw):
    kv_len = kw.pop("kv_len", None)
    lat_edit = kw.pop("lat_edit", None)
    calls = kw.pop("calls", False)
    persistent = kw.pop("persistent", False)
    edit = kw.pop("edit", None)             # edit(inp, tree): after the tree is known
    inp, tree_o = prepare(scfg, seed, kv_len=kv_len, lat_edit=lat_edit)
    if edit is not None:
        edit(inp, tree_o)
    st = run_gpu(scfg, inp, calls=calls, persistent=persistent)
    res = compare(scfg, inp, tree_o, st, **kw)
    res["status"] = __import__("speculative_decoding_tree_best_gb300.binding",
                               fromlist=["x"]).spec_status_read(st.ws)
    return res
