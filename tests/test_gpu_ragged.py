"""GPU parity of the batch that shares a node budget (per-request draft
positions, best-first over all requests' frontiers): trees bit-exact against
the oracle, and the whole fused step over those trees."""
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


def _trees(scfg, seed, m_req, budget, ties=False):
    inp = synth.make_step_inputs(scfg, seed, logits=False)
    if ties:
        inp["lat_score"] = (-0.5 * torch.randint(0, 3, inp["lat_score"].shape,
                                                 generator=torch.Generator().manual_seed(seed))
                            ).float().contiguous()
    m_req = torch.as_tensor(m_req, dtype=torch.int32)
    want = oracle.tree_build_ragged(inp["lat_tok"], inp["lat_score"], inp["root_tok"], scfg.N,
                                    m_req, budget)
    cfg = binding.make_cfg(scfg)
    tree = binding.TreeBuffers(cfg)
    ws = binding.alloc_workspace(cfg)
    binding.spec_tree_build_ragged(cfg, inp["lat_tok"].cuda(), inp["lat_score"].cuda(),
                                   inp["root_tok"].cuda(), m_req.cuda(), budget, tree, ws)
    torch.cuda.synchronize()
    got = tree.to_numpy()
    for k in ("n_nodes", "node_tok", "node_parent", "node_depth", "node_rank", "node_anc"):
        np.testing.assert_array_equal(got[k], want[k], err_msg=k)
    np.testing.assert_array_equal(got["node_score"].view(np.uint32),
                                  want["node_score"].view(np.uint32), err_msg="node_score bits")
    return binding.spec_status_read(ws), want


SMALL = synth.config(1).replace(B=5, m=6, K=4, N=12, V=500, L=300)


@pytest.mark.parametrize("budget", [-1, 0, 1, 7, 23, 60, 1000])
def test_trees_with_shared_budget(budget):
    status, want = _trees(SMALL, 3, [6, 4, 2, 1, 5], budget)
    assert status == 0
    if budget >= 0:
        assert int((want["n_nodes"] - 1).sum()) <= budget


def test_trees_with_tied_scores():
    for budget in (-1, 9, 25):
        _trees(SMALL.replace(K=6), 4, [6, 6, 3, 3, 1], budget, ties=True)


def test_ragged_workload_trees_full_size():
    scfg = synth.config(5)
    status, want = _trees(scfg, 0, scfg.m_req(), scfg.budget)
    assert status == 0 and int((want["n_nodes"] - 1).sum()) == 192


def test_out_of_range_positions_are_clamped_and_reported():
    inp = synth.make_step_inputs(SMALL, 5, logits=False)
    cfg = binding.make_cfg(SMALL)
    tree = binding.TreeBuffers(cfg)
    ws = binding.alloc_workspace(cfg)
    m_req = torch.tensor([0, 9, 3, 6, 1], dtype=torch.int32)
    binding.spec_tree_build_ragged(cfg, inp["lat_tok"].cuda(), inp["lat_score"].cuda(),
                                   inp["root_tok"].cuda(), m_req.cuda(), -1, tree, ws)
    assert binding.spec_status_read(ws) & binding.SPEC_DEV_BADREQ
    clamped = torch.tensor([1, 6, 3, 6, 1], dtype=torch.int32)
    want = oracle.tree_build_ragged(inp["lat_tok"], inp["lat_score"], inp["root_tok"], SMALL.N,
                                    clamped, -1)
    np.testing.assert_array_equal(tree.to_numpy()["node_tok"], want["node_tok"])


def test_fused_step_over_ragged_trees():
    scfg = synth.config(5).replace(B=6, V=3000, L=400, L_lo=50, budget=30)
    r = parity.check_case(scfg, 1)
    assert r["status"] == 0
    r = parity.check_case(scfg, 2, calls=True)
    assert r["status"] == 0


def test_ragged_workload_step_sampled():
    r = parity.check_case(synth.config(5), 0, req=[0, 1, 2, 13], attn_kv_heads=[1, 6])
    assert r["status"] == 0
