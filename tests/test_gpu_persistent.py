"""GPU parity of the persistent verify + commit (one cooperative launch for the
argmax, the acceptance, the KV append and every GDN layer's verify + commit
from the state held in shared memory) against the oracle, and against the
unfused step on the same inputs."""
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


SMALL = synth.config(1).replace(m=4, K=4, N=12, L=300, V=4096)


@pytest.mark.parametrize("seed", range(3))
def test_single_request_full_size(seed):
    r = parity.check_case(synth.config(1), seed, persistent=True)
    assert r["status"] == 0


def test_batched_sampled():
    r = parity.check_case(synth.config(3), 1, persistent=True, req=[0, 11, 23],
                          attn_kv_heads=[1, 6])
    assert r["status"] == 0


def test_multi_layer_stack_small():
    cfg = synth.config(4).replace(B=2, n_gdn=3, n_attn=2, L=257, V=3000)
    assert parity.check_case(cfg, 9, persistent=True)["status"] == 0


def test_no_attention_layers():
    # the tree is then the launch right before the fused one
    assert parity.check_case(SMALL.replace(n_attn=0), 2, persistent=True)["status"] == 0


def test_cache_overflow_leaves_the_state():
    cfg = SMALL.replace(B=2, L=200, headroom=0)
    r = parity.check_case(cfg, 7, kv_len=[200, 10], persistent=True)
    assert r["overflow"] == [True, False]
    assert r["status"] & binding.SPEC_DEV_OVERFLOW


def test_padding_rows_and_single_row_tree():
    parity.check_case(SMALL.replace(m=2, K=2, N=20), 3, persistent=True)
    parity.check_case(SMALL.replace(N=0), 4, persistent=True)


def _pair(cfg, seed):
    from speculative_decoding_tree_best_gb300.step import VerifyStep, stack_inputs
    inp, _ = parity.prepare(cfg, seed)
    return (VerifyStep(cfg, stack_inputs(inp, "cuda"), persistent=True),
            VerifyStep(cfg, stack_inputs(inp, "cuda")))


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


@pytest.mark.parametrize("ci", [1, 4])
def test_same_results_as_the_unfused_step_over_three_steps(ci):
    """Trees, attention outputs, acceptance and KV commits bit-identical to
    spec_verify_step, GDN outputs and committed states within float rounding,
    three steps in a row (a queue, ticket or flag left set would break the
    next step)."""
    cfg = synth.config(1) if ci == 1 else synth.config(4).replace(B=3, n_gdn=2, n_attn=2, L=300)
    p, u = _pair(cfg, 5)
    assert p.launches_per_step == 1 + 2 * cfg.n_attn + 1
    for step in range(3):
        p.run()
        u.run()
        torch.cuda.synchronize()
        for k in ("node_tok", "node_parent", "node_score", "n_nodes"):
            assert torch.equal(getattr(p.tree, k), getattr(u.tree, k)), (step, k)
        assert torch.equal(p.attn_o, u.attn_o), step
        # the same sums in another rounding order (and, after the first step,
        # states committed by another exact formula); the two GDN kernels also
        # split the fp32 state into bf16 terms differently (rounded or
        # truncated high term), so a few bf16 outputs round the other way
        assert _rel(p.gdn_o, u.gdn_o) < 1e-3, step
        for k in ("argmax", "accept_len", "accept_nodes", "out_tok"):
            assert torch.equal(getattr(p.acc, k), getattr(u.acc, k)), (step, k)
        for k in ("k_cache", "v_cache", "kv_len", "root_tok"):
            assert torch.equal(p.x[k], u.x[k]), (step, k)
        assert _rel(p.x["gdn_h0"], u.x["gdn_h0"]) < 1e-5, step
        assert binding.spec_status_read(p.ws) == 0
