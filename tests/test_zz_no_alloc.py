"""attn_tree_verify_noalloc (static library scratch, no workspace) against
attn_tree_verify (caller workspace) on the same inputs: two calls in a row,
each within the parity tolerance of the workspace call (the same kernels run,
so the results are expected to be identical).  Collected last so that it also
runs after every other GPU test in the same process."""
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


def _attn_inputs(scfg, seed):
    from speculative_decoding_tree_best_gb300.step import stack_inputs
    inp, _ = parity.prepare(scfg, seed)
    x = stack_inputs(inp, "cuda")
    cfg = binding.make_cfg(scfg)
    tree = binding.TreeBuffers(cfg)
    ws = binding.alloc_workspace(cfg)
    binding.spec_tree_build(cfg, x["lat_tok"], x["lat_score"], x["root_tok"], tree, ws)
    a = {k: x[k][0].contiguous() for k in ("attn_q", "k_tree", "v_tree", "k_cache", "v_cache")}
    return cfg, tree, ws, a, x["kv_len"]


@pytest.mark.parametrize("ci,seed", [(1, 0), (0, 1)])
def test_noalloc_matches_workspace_call_twice(ci, seed):
    scfg = synth.config(ci)
    cfg, tree, ws, a, kv_len = _attn_inputs(scfg, seed)
    args = (a["attn_q"], a["k_tree"], a["v_tree"], a["k_cache"], a["v_cache"], kv_len)
    want = torch.empty_like(a["attn_q"])
    binding.attn_tree_verify(cfg, tree, *args, want, ws)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        got = torch.full_like(a["attn_q"], float("nan"))
        binding.attn_tree_verify_noalloc(cfg, tree, *args, got, status)
        torch.cuda.synchronize()
        e = parity.rel_l2(got.double().cpu().numpy(), want.double().cpu().numpy())
        assert e <= parity.REL_L2, f"rel-L2 {e:.3e} against attn_tree_verify"
        assert torch.isfinite(got).all()
    assert int(status.item()) == 0
    assert binding.spec_status_read(ws) == 0


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    """24 requests with an 8K cache need ~57 MB of partials: rejected on the
    host before any device work (the small buffers below are never read)."""
    cfg = binding.make_cfg(synth.config(3))
    tree = binding.TreeBuffers(cfg)
    small = [torch.zeros(64, dtype=torch.bfloat16, device="cuda") for _ in range(6)]
    kv_len = torch.zeros(cfg.B, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.SpecError) as ei:
        binding.attn_tree_verify_noalloc(cfg, tree, *small[:5], kv_len, small[5])
    assert ei.value.code == binding.ST_ESCRATCH
