"""GPU parity of the Markov-head tree builder: the edge scores depend on the
parent's token (l = base + <W1[x], W2[y]>, minus the log-sum-exp over the
position's candidates), fixed to the bit by their fp32 algorithm; trees are
compared bit for bit with the oracle."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_best_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_best_gb300 import build
    build.build()
    binding.load()


def _check(scfg, seed, R=32, zero=False, ties=False):
    g = torch.Generator().manual_seed(seed)
    lat_tok, _, root = synth.make_lattice(scfg, g)
    base, W1, W2 = synth.make_markov(scfg, g, R)
    if zero:
        W1.zero_()
        W2.zero_()
    if ties:
        base = (-0.5 * torch.randint(0, 3, base.shape, generator=g)).float().contiguous()
    want = oracle.tree_build_markov(lat_tok, base, W1, W2, root, scfg.N)
    cfg = binding.make_cfg(scfg)
    tree = binding.TreeBuffers(cfg)
    ws = binding.alloc_workspace(cfg)
    binding.spec_tree_build_markov(cfg, lat_tok.cuda(), base.cuda(), W1.cuda(), W2.cuda(),
                                   root.cuda(), tree, ws)
    torch.cuda.synchronize()
    got = tree.to_numpy()
    for k in ("n_nodes", "node_tok", "node_parent", "node_depth", "node_rank", "node_anc"):
        np.testing.assert_array_equal(got[k], want[k], err_msg=k)
    np.testing.assert_array_equal(got["node_score"].view(np.uint32),
                                  want["node_score"].view(np.uint32), err_msg="node_score bits")
    assert binding.spec_status_read(ws) == 0
    return want


SMALL = synth.config(1).replace(B=3, m=4, K=6, N=20, V=300)


@pytest.mark.parametrize("seed", range(4))
def test_small_lattices(seed):
    _check(SMALL, seed, R=8)


def test_single_request_shape():
    for seed in range(3):
        _check(synth.config(1), seed)


def test_long_tree_two_slots_per_lane():
    _check(synth.config(2), 0)                 # 16 positions, N = 64


def test_batched_requests():
    _check(synth.config(3).replace(L=600, L_lo=100), 1)


def test_zero_head_and_tied_bases():
    _check(SMALL.replace(K=8), 5, R=4, zero=True, ties=True)
    _check(SMALL, 6, R=0)


@pytest.mark.parametrize("R", [1, 7, 33])
def test_head_ranks_not_a_multiple_of_four(R):
    _check(SMALL, 10 + R, R=R)                 # the 4-byte staging path


@pytest.mark.parametrize("K", [17, 32])
def test_wide_positions_use_full_warps(K):
    _check(SMALL.replace(K=K), 20 + K, R=12)


def test_out_of_range_token_is_reported_and_stays_local():
    scfg = SMALL
    g = torch.Generator().manual_seed(7)
    lat_tok, _, root = synth.make_lattice(scfg, g)
    base, W1, W2 = synth.make_markov(scfg, g, 8)
    want = oracle.tree_build_markov(lat_tok, base, W1, W2, root, scfg.N)
    bad_tok = lat_tok.clone()
    bad_tok[1, 2, 3] = scfg.V                  # one past the head's last row
    cfg = binding.make_cfg(scfg)
    tree = binding.TreeBuffers(cfg)
    ws = binding.alloc_workspace(cfg)
    binding.spec_tree_build_markov(cfg, bad_tok.cuda(), base.cuda(), W1.cuda(), W2.cuda(),
                                   root.cuda(), tree, ws)
    torch.cuda.synchronize()
    assert binding.spec_status_read(ws) & binding.SPEC_DEV_BADLAT
    got = tree.to_numpy()
    for b in (0, 2):                           # the other requests are untouched
        for k in ("node_tok", "node_parent", "node_rank"):
            np.testing.assert_array_equal(got[k][b], want[k][b], err_msg=k)


def test_fused_step_with_markov_head():
    from tests import parity
    scfg = synth.config(6).replace(V=3000, L=500)
    assert parity.check_case(scfg, 0)["status"] == 0
    assert parity.check_case(scfg, 1, calls=True)["status"] == 0


def test_markov_workload_step():
    from tests import parity
    assert parity.check_case(synth.config(6), 2)["status"] == 0
