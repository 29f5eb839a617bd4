"""GPU parity of the sampled acceptance (temperature > 0): each row's draw, the
walk over the draws and the commit, against the oracle on the same seeded
inputs (draws bit-exact except rows whose top-2 score gap is below 1e-3)."""
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


SAMPLED = synth.config(7)
SMALL = SAMPLED.replace(V=10000, L=300)                # three chunks, the last one ragged


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("calls", [False, True])
def test_small_vocabulary(seed, calls):
    r = parity.check_case(SMALL, seed, calls=calls)
    assert r["status"] == 0


def test_fp32_io_one_chunk():
    scfg = synth.config(0).replace(temperature=0.7, sample_seed=77, plant_gap=8.0)
    for seed in range(3):
        assert parity.check_case(scfg, seed)["status"] == 0
        assert parity.check_case(scfg, seed, calls=True)["status"] == 0


def test_vocabulary_not_a_multiple_of_the_vector_width():
    r = parity.check_case(SMALL.replace(V=9999), 4)      # the 2-byte load path
    assert r["status"] == 0


@pytest.mark.parametrize("temperature", [0.3, 2.0])
def test_other_temperatures(temperature):
    assert parity.check_case(SMALL.replace(temperature=temperature), 5)["status"] == 0


def test_batched_requests_and_positions():
    scfg = SMALL.replace(B=6, L=400, L_lo=50)
    r = parity.check_case(scfg, 6)
    assert r["status"] == 0


def test_sampled_workload_step():
    r = parity.check_case(SAMPLED, 0)
    assert r["status"] == 0
    assert max(r["tau"]) >= 2                      # the planted rows do get accepted


def test_steps_without_attention_layers():
    # the tree is then the launch right before the acceptance
    for scfg in (SMALL.replace(n_attn=0), SMALL.replace(n_attn=0, temperature=0.0)):
        assert parity.check_case(scfg, 8)["status"] == 0


def test_row_without_a_finite_score_is_reported():
    inp, _ = parity.prepare(SMALL, 9)
    inp["logits"][0, 0, :] = float("nan")
    st = parity.run_gpu(SMALL, inp, calls=True)
    assert binding.spec_status_read(st.ws) & binding.SPEC_DEV_BADLOGIT
    assert 0 <= int(st.acc.argmax[0, 0]) < SMALL.V
