"""attn_tree_verify_noalloc (the library's static scratch, no workspace)
against the CPU oracle and against attn_tree_verify (caller workspace) on the
same inputs: two calls in a row, each within the parity bound of the oracle
and bit-identical to the workspace call (the same kernels run); the largest
cache the 8 MiB scratch holds for one request, and one row more, which is
refused.  Collected last so that it also runs after every other GPU test in
the same process."""
import numpy as np
import pytest
import torch

import oracle
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


def _attn_inputs(scfg, seed, kv_len=None):
    from speculative_decoding_tree_best_gb300.step import stack_inputs
    inp, tree_o = parity.prepare(scfg, seed, kv_len=kv_len)
    x = stack_inputs(inp, "cuda")
    cfg = binding.make_cfg(scfg)
    tree = binding.TreeBuffers(cfg)
    ws = binding.alloc_workspace(cfg)
    binding.spec_tree_build(cfg, x["lat_tok"], x["lat_score"], x["root_tok"], tree, ws)
    a = {k: x[k][0].contiguous() for k in ("attn_q", "k_tree", "v_tree", "k_cache", "v_cache")}
    return cfg, tree, ws, a, x["kv_len"], inp, tree_o


def _check_against_oracle(scfg, inp, tree_o, got, kv_heads):
    """got [B][T][Hq][D] against the oracle on the q-heads of `kv_heads`:
    whole-tensor and per-row rel-L2 bounds of the parity contract, zero
    padding rows."""
    G = scfg.Hq // scfg.Hkv
    qh = [g * G + i for g in kv_heads for i in range(G)]
    lay = inp["attn"][0]
    want = oracle.attn_tree({k: tree_o[k] for k in ("n_nodes", "node_anc")},
                            lay["q"][:, :, qh].contiguous(), lay["k_tree"][:, :, kv_heads].contiguous(),
                            lay["v_tree"][:, :, kv_heads].contiguous(),
                            lay["k_cache"][:, :, kv_heads].contiguous(),
                            lay["v_cache"][:, :, kv_heads].contiguous(), inp["kv_len"])
    g = got[:, :, qh].double().cpu().numpy()
    nn = tree_o["n_nodes"]
    for b in range(scfg.B):
        assert not g[b, nn[b]:].any(), "padding rows must be zero"
    e = parity.rel_l2(g, want)
    assert e <= parity.REL_L2, f"rel-L2 {e:.3e} against the oracle"
    valid = np.zeros(g.shape[:3], bool)
    for b in range(scfg.B):
        valid[b, :nn[b]] = True
    er, at = parity.row_rel_l2(g, want, valid)
    assert er <= parity.ROW_REL_L2, f"row {at} rel-L2 {er:.3e} against the oracle"


def _two_calls(cfg, tree, ws, a, kv_len):
    args = (a["attn_q"], a["k_tree"], a["v_tree"], a["k_cache"], a["v_cache"], kv_len)
    want = torch.empty_like(a["attn_q"])
    binding.attn_tree_verify(cfg, tree, *args, want, ws)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):
        got = torch.full_like(a["attn_q"], float("nan"))
        binding.attn_tree_verify_noalloc(cfg, tree, *args, got, status)
        torch.cuda.synchronize()
        assert torch.equal(got, want), "no-allocation call differs from attn_tree_verify"
        outs.append(got)
    assert int(status.item()) == 0
    assert binding.spec_status_read(ws) == 0
    return outs[-1]


@pytest.mark.parametrize("ci,seed", [(1, 0), (0, 1)])
def test_noalloc_matches_oracle_and_workspace_call_twice(ci, seed):
    scfg = synth.config(ci)
    cfg, tree, ws, a, kv_len, inp, tree_o = _attn_inputs(scfg, seed)
    got = _two_calls(cfg, tree, ws, a, kv_len)
    _check_against_oracle(scfg, inp, tree_o, got, list(range(scfg.Hkv)))


# One request, 8 kv-heads of 128, T = 25, bf16: the partials take
# 8 heads x 31 chunks of 2048 keys (30 cache chunks + the tree chunk) x 128
# rows x (128 fp16 + 2 floats) = 8.38 MB of the 8 MiB scratch at Lmax = 61440;
# one row more needs a 31st cache chunk (8.65 MB).  Keys come in chunks of 2048
# at this length on any device of up to 240 SMs.
LMAX_FITS = 61440


def test_noalloc_largest_cache_that_fits():
    """Lmax = 61440 fits: a KV length of 61000 writes partials into the last
    cache chunk (the end of the scratch); oracle parity on two kv-heads, and
    bit-identical to the workspace call."""
    scfg = synth.config(1).replace(L=LMAX_FITS - 64, headroom=64)
    assert scfg.Lmax == LMAX_FITS
    cfg, tree, ws, a, kv_len, inp, tree_o = _attn_inputs(scfg, 2, kv_len=[61000])
    got = _two_calls(cfg, tree, ws, a, kv_len)
    _check_against_oracle(scfg, inp, tree_o, got, [0, 7])


def _refused(scfg):
    cfg = binding.make_cfg(scfg)
    tree = binding.TreeBuffers(cfg)
    small = [torch.zeros(64, dtype=torch.bfloat16, device="cuda") for _ in range(6)]
    kv_len = torch.zeros(cfg.B, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.SpecError) as ei:
        binding.attn_tree_verify_noalloc(cfg, tree, *small[:5], kv_len, small[5])
    assert ei.value.code == binding.ST_ESCRATCH


def test_noalloc_rejects_one_row_past_the_scratch():
    """Lmax = 61441 is refused on the host before any device work (the small
    buffers passed are never read)."""
    _refused(synth.config(1).replace(L=LMAX_FITS + 1 - 64, headroom=64))


def test_noalloc_rejects_a_large_batch():
    """24 requests with an 8K cache need ~57 MB of partials: refused."""
    _refused(synth.config(3))
