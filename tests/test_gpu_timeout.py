"""A bounded device wait that nothing satisfies ends with SPEC_DEV_TIMEOUT in
the status word, the kernel returns, and the context stays usable: the next
verify step still matches the oracle.  (No trap, fault or hang is involved.)"""
import time

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


def test_satisfied_wait_leaves_status_clear():
    ws = binding.alloc_workspace(binding.make_cfg(synth.config(0)))
    binding.spec_wait_probe(2000, True, ws)
    assert binding.spec_status_read(ws) == 0


def test_unsatisfied_wait_times_out_and_context_survives():
    ws = binding.alloc_workspace(binding.make_cfg(synth.config(0)))
    t0 = time.perf_counter()
    binding.spec_wait_probe(20000, False, ws)          # ~20 ms limit
    st = binding.spec_status_read(ws)                  # synchronises the stream
    assert st & binding.SPEC_DEV_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    binding.spec_status_clear(ws)
    assert binding.spec_status_read(ws) == 0
    r = parity.check_case(synth.config(0), 11)         # the context is still usable
    assert r["status"] == 0
