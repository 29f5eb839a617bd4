"""GPU parity: the CUDA library, called through its C ABI, against the CPU
oracle on the same seeded inputs (bit-exact on trees, argmax, acceptance and
commits; rel-L2 <= 2e-3 on GDN/attention outputs and committed states)."""
import pytest
import torch

from speculative_decoding_tree_best_gb300 import binding, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_best_gb300 import build
    build.build()
    binding.load()


@pytest.mark.parametrize("seed", range(5))
def test_tiny_fp32(seed):
    r = parity.check_case(synth.config(0), seed, calls=seed % 2 == 1)
    assert r["gdn_rel_l2"] < 1e-5 and r["attn_rel_l2"] < 1e-5 and r["state_rel_l2"] < 1e-5
    assert r["status"] == 0


@pytest.mark.parametrize("seed", range(3))
def test_single_request_full_size(seed):
    r = parity.check_case(synth.config(1), seed, calls=seed == 2)
    assert r["status"] == 0


@pytest.mark.parametrize("ci", [1, 4])
def test_fused_step_equals_the_four_calls(ci):
    """spec_verify_step and the four calls in order give identical bits."""
    from speculative_decoding_tree_best_gb300.step import VerifyStep, stack_inputs
    cfg = synth.config(ci) if ci == 1 else synth.config(4).replace(B=2, n_gdn=3, n_attn=3, L=300)
    inp, _ = parity.prepare(cfg, 3)
    a = VerifyStep(cfg, stack_inputs(inp, "cuda"))
    b = VerifyStep(cfg, stack_inputs(inp, "cuda"))
    a.run()
    b.run_calls()
    torch.cuda.synchronize()
    # tree, partials + merges per attention layer, argmax + acceptance (in the
    # last merge's launch for at most 64 logits rows), one launch per GDN
    # layer, commit
    merged = cfg.B * cfg.T <= 64
    assert a.launches_per_step == 1 + 2 * cfg.n_attn + (0 if merged else 1) + cfg.n_gdn + 1
    for k in ("node_tok", "node_parent", "node_depth", "node_rank", "node_score", "node_anc",
              "n_nodes"):
        assert torch.equal(getattr(a.tree, k), getattr(b.tree, k)), k
    assert torch.equal(a.gdn_o, b.gdn_o) and torch.equal(a.attn_o, b.attn_o)
    for k in ("argmax", "accept_len", "accept_nodes", "out_tok"):
        assert torch.equal(getattr(a.acc, k), getattr(b.acc, k)), k
    for k in ("gdn_h0", "k_cache", "v_cache", "kv_len", "root_tok"):
        assert torch.equal(a.x[k], b.x[k]), k


def test_long_tree_full_size_sampled():
    r = parity.check_case(synth.config(2), 0, attn_kv_heads=[0, 5])
    assert max(r["tau"]) >= 1


def test_batched_sampled():
    r = parity.check_case(synth.config(3), 0, req=[0, 7, 23], attn_kv_heads=[2, 7])
    assert r["status"] == 0


# ---- edge cases ---------------------------------------------------------------------

SMALL = synth.config(1).replace(m=4, K=4, N=12, L=300, V=4096)


def test_single_row_tree():
    parity.check_case(SMALL.replace(N=0), 1)


def test_frontier_exhausted_padding_rows():
    r = parity.check_case(SMALL.replace(m=2, K=2, N=20), 2)     # 6 drafts exist, 14 pad rows
    assert r["status"] == 0


def test_k1_chain_and_m1_star():
    parity.check_case(SMALL.replace(K=1, N=6), 3)
    parity.check_case(SMALL.replace(m=1, K=16, N=10), 4)


def test_tied_lattice_scores():
    def ties(inp):
        inp["lat_score"] = (-0.5 * torch.randint(0, 3, inp["lat_score"].shape,
                                                 generator=torch.Generator().manual_seed(0))
                            ).float().contiguous()
    parity.check_case(SMALL.replace(m=4, K=8, N=40), 5, lat_edit=ties)


def test_empty_cache_and_ragged_lengths():
    cfg = SMALL.replace(B=4, L=700, N=12)
    parity.check_case(cfg, 6, kv_len=[0, 1, 129, 700])


def test_cache_overflow_skips_commit():
    cfg = SMALL.replace(B=2, L=200, headroom=0)
    r = parity.check_case(cfg, 7, kv_len=[200, 10])
    assert r["overflow"] == [True, False]
    assert r["status"] & binding.SPEC_DEV_OVERFLOW


def test_head_dim_64_bf16_and_deep_tree():
    cfg = synth.config(1).replace(dk=64, dv=64, D=64, Hk=4, Hv=8, Hq=8, Hkv=2, m=16, K=4,
                                  N=100, L=513, V=2000)
    parity.check_case(cfg, 8)


def test_multi_layer_stack_small():
    cfg = synth.config(4).replace(B=2, n_gdn=3, n_attn=2, L=257, V=3000)
    parity.check_case(cfg, 9)
    parity.check_case(cfg, 10, calls=True)


def test_full_stack_sampled():
    """The 64-layer stack at full size (8 requests, 48 GDN + 16 attention
    layers, KV 8192) in the launch configuration the bench times: every tree,
    argmax, acceptance and kv_len bit for bit; the floats of the first and last
    layer of each kind, for two requests and one kv-head group."""
    r = parity.check_case(synth.config(4), 0, req=[0, 5], attn_kv_heads=[3], gdn_layers=[0, 47],
                          attn_layers=[0, 15])
    assert r["status"] == 0 and min(r["tau"]) >= 1


def test_repeated_batched_attention_no_timeout():
    """Sixty batched attention launches in a row (the persistent partial runs
    several units per CTA with its rings crossing unit boundaries): every
    bounded wait completes (no timeout bit) and every launch gives the same
    bits."""
    from speculative_decoding_tree_best_gb300.step import VerifyStep, stack_inputs
    cfg = synth.config(3)
    inp, _ = parity.prepare(cfg, 4)
    st = VerifyStep(cfg, stack_inputs(inp, "cuda"))
    st.build_tree()
    x, c = st.x, st.cfg

    def attn():
        binding.attn_tree_verify(c, st.tree, x["attn_q"][0], x["k_tree"][0], x["v_tree"][0],
                                 x["k_cache"][0], x["v_cache"][0], x["kv_len"], st.attn_o[0],
                                 st.ws)
    attn()
    torch.cuda.synchronize()
    first = st.attn_o.clone()
    for _ in range(60):
        attn()
    torch.cuda.synchronize()
    assert binding.spec_status_read(st.ws) == 0
    assert torch.equal(st.attn_o, first)


@pytest.mark.parametrize("dk,dv", [(128, 64), (64, 128)])
def test_unequal_key_and_value_head_dims(dk, dv):
    parity.check_case(SMALL.replace(dk=dk, dv=dv, Hk=2, Hv=4), 11)


@pytest.mark.parametrize("N", [90, 95])
def test_trees_with_a_full_third_row_slot(N):
    """Trees of 91 and 96 rows: the tree builder's third 32-row slot then
    holds many rows (a parent and its new child both there, on different
    lanes); bit-exact like every tree, and the step around them at parity."""
    parity.check_case(SMALL.replace(m=8, K=16, N=N), 12 + N % 2)


def _inf_where_unread(inp, tree_o):
    """inf in every input row the step must not read: cache rows at or past
    kv_len, and the tree-row inputs (and gates) of the padding rows."""
    nn = tree_o["n_nodes"]
    inf = float("inf")
    for b in range(len(nn)):
        L, n = int(inp["kv_len"][b]), int(nn[b])
        for lay in inp["attn"]:
            lay["k_cache"][b, L:] = inf
            lay["v_cache"][b, L:] = inf
            for k in ("q", "k_tree", "v_tree"):
                lay[k][b, n:] = inf
        for lay in inp["gdn"]:
            for k in ("q", "k", "v", "alpha", "beta"):
                lay[k][b, n:] = inf


@pytest.mark.parametrize("case", ["tiny_fp32", "bf16", "bf16_persistent", "bf16_long_tree"])
def test_rows_outside_the_valid_ranges_are_never_read(case):
    """Results do not depend on cache rows at or past kv_len, nor on the
    padding rows of the tree-row inputs: with inf in all of them (0 x inf is
    NaN, so a masked product over them would show) every output matches the
    oracle, which never reads them, and no status bit is raised."""
    if case == "tiny_fp32":
        cfg, kv, kw = synth.config(0).replace(N=12, L=200), None, {}
    else:
        cfg = SMALL.replace(B=2, L=700, N=40 if case == "bf16_long_tree" else 20, m=4, K=8)
        kv, kw = [650, 333], {"persistent": case == "bf16_persistent"}
    r = parity.check_case(cfg, 14, kv_len=kv, edit=_inf_where_unread, **kw)
    assert r["status"] == 0


@pytest.mark.parametrize("where,value,flagged", [("cache", 7.0e4, True), ("tree", 7.0e4, True),
                                                 ("cache", 6.5e4, False)])
def test_v_beyond_fp16_range_is_flagged(where, value, flagged):
    """The attention's P.V product takes V in fp16: a visible bf16 V value of
    7e4 (beyond fp16's 65504) in request 1 raises SPEC_DEV_RANGE and makes its
    outputs non-finite, while request 0 still matches the oracle; 6.5e4 is in
    range, raises nothing, and both requests match."""
    cfg = SMALL.replace(B=2, L=700)
    inp, tree_o = parity.prepare(cfg, 13, kv_len=[650, 333])
    lay = inp["attn"][0]
    if where == "cache":
        lay["v_cache"][1, 100, 3, 17] = value
    else:
        lay["v_tree"][1, 0, 3, 17] = value          # the root row: every row sees it
    st = parity.run_gpu(cfg, inp)
    status = binding.spec_status_read(st.ws)
    G = cfg.Hq // cfg.Hkv
    if flagged:
        assert status & binding.SPEC_DEV_RANGE
        assert not torch.isfinite(st.attn_o[0][1, :, 3 * G:4 * G].float()).all()
        parity.compare(cfg, inp, tree_o, st, req=[0])
    else:
        assert status == 0
        parity.compare(cfg, inp, tree_o, st)


@pytest.mark.parametrize("ci", [1, 4])
def test_host_step_equals_the_device_step(ci):
    """step.HostStep (inputs copied from pinned host memory in pieces on a copy
    stream, each phase waiting for its own piece, captured as a graph) gives
    the same bits as the fused step on device-resident inputs: after its eager
    first run and after a graph replay (two consecutive steps)."""
    from speculative_decoding_tree_best_gb300.step import HostStep, VerifyStep, stack_inputs
    cfg = synth.config(ci) if ci == 1 else synth.config(4).replace(B=2, n_gdn=3, n_attn=2, L=300)
    inp, _ = parity.prepare(cfg, 3)
    a = VerifyStep(cfg, stack_inputs(inp, "cuda"))
    b = VerifyStep(cfg, stack_inputs(inp, "cuda"))
    hs = HostStep(b)
    for rep in range(2):
        a.run()
        if rep == 0:
            hs.capture()          # runs the sequence once, then captures it
        else:
            hs.run()
        torch.cuda.synchronize()
        for k in ("node_tok", "node_parent", "node_anc", "n_nodes"):
            assert torch.equal(getattr(a.tree, k), getattr(b.tree, k)), k
        assert torch.equal(a.gdn_o, b.gdn_o) and torch.equal(a.attn_o, b.attn_o)
        for k in ("argmax", "accept_len", "accept_nodes", "out_tok"):
            assert torch.equal(getattr(a.acc, k), getattr(b.acc, k)), k
        for k in ("gdn_h0", "k_cache", "v_cache", "kv_len", "root_tok"):
            assert torch.equal(a.x[k], b.x[k]), k
        assert torch.equal(hs.out["accept_len"], a.acc.accept_len.cpu())
        assert torch.equal(hs.out["out_tok"], a.acc.out_tok.cpu())
