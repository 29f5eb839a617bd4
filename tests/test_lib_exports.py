"""The C-ABI library builds, loads and exports every function spec_tree.h
declares; host-side argument validation rejects bad input before any CUDA
call.  Runs without a GPU (no kernel is launched here)."""
import ctypes
import os
import re
import shutil

import pytest

from speculative_decoding_tree_best_gb300 import binding, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_tree.h")


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from speculative_decoding_tree_best_gb300 import build
    build.build()
    return binding.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\([^;]*\)\s*;", src, re.M)))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("spec_tree_build", "gdn_tree_verify", "attn_tree_verify", "accept_and_commit",
              "spec_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in spec_tree.h but not exported"
    assert set(binding.EXPORTS) <= set(declared_functions())


def test_abi_version_and_strings(lib):
    assert lib.spec_abi_version() == 1
    for code in range(6):
        assert lib.spec_status_string(code)


def test_workspace_sizing_is_host_only(lib):
    for i in range(5):
        cfg = binding.make_cfg(synth.config(i))
        n = binding.spec_workspace_bytes_for_sms(cfg, 152)
        assert n > 256 and n % 256 == 0
    bad = binding.make_cfg(synth.config(1), dk=96)
    assert lib.spec_workspace_bytes(ctypes.byref(bad)) == 0
    assert lib.spec_workspace_bytes_for_sms(ctypes.byref(bad), 152) == 0
    assert lib.spec_workspace_bytes_for_sms(ctypes.byref(binding.make_cfg(synth.config(1))), 0) == 0


def test_workspace_layout_follows_the_sm_count(lib):
    """The attention's keys are cut into about one chunk per SM for small
    problems: a single request's 4096-key cache gives 256-key chunks on 152
    SMs but 2048-key chunks on 16, so the split-KV partials shrink; 24 requests
    already fill the device with 2048-key chunks at either count."""
    one = binding.make_cfg(synth.config(1))
    assert binding.spec_workspace_bytes_for_sms(one, 16) < binding.spec_workspace_bytes_for_sms(one, 152)
    # 152 SMs: 17 chunks of 256 keys + the tree chunk, 8 kv-heads x 1 tile, fp16
    # partials [..][128][128] and (max, sum) [..][128]
    tiles = 8 * (16 + 1)
    assert binding.spec_workspace_bytes_for_sms(one, 152) >= tiles * 128 * (128 * 2 + 8)
    many = binding.make_cfg(synth.config(3))
    assert (binding.spec_workspace_bytes_for_sms(many, 132)
            == binding.spec_workspace_bytes_for_sms(many, 152))


def test_step_launch_count_is_host_only(lib):
    # tree, attention partials + merge, argmax/accept, GDN, commit
    # tree, partials + merges, argmax (in the last merge's launch for at most
    # 64 logits rows), GDN, commit
    assert binding.spec_step_launches(binding.make_cfg(synth.config(0))) == 5
    assert binding.spec_step_launches(binding.make_cfg(synth.config(1))) == 5
    assert binding.spec_step_launches(binding.make_cfg(synth.config(3))) == 6
    assert binding.spec_step_launches(binding.make_cfg(synth.config(4))) == 1 + 32 + 1 + 48 + 1
    # without attention layers the argmax is a launch of its own
    assert binding.spec_step_launches(binding.make_cfg(synth.config(1).replace(n_attn=0))) == 4
    bad = binding.make_cfg(synth.config(1), dk=96)
    assert lib.spec_step_launches(ctypes.byref(bad)) == -1


def test_shared_budget_beyond_one_cta_is_unsupported(lib):
    """The budget step holds every score of the batch in one CTA's shared
    memory; larger batches are refused on the host before any launch."""
    cfg = binding.make_cfg(synth.config(1), B=2000, N=127)
    rc = lib.spec_tree_build_ragged(ctypes.byref(cfg), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                    ctypes.c_void_p(16), None, 100,
                                    ctypes.byref(binding.SpecTree(*([16] * 7))),
                                    ctypes.c_void_p(16), None)
    assert rc == binding.ST_EUNSUPPORTED


@pytest.mark.parametrize("field,value", [("K", 33), ("N", 128), ("m", 0), ("Hv", 20),
                                         ("Hq", 30), ("D", 256), ("io_dtype", 7)])
def test_validation_rejects_before_launch(lib, field, value):
    cfg = binding.make_cfg(synth.config(1), **{field: value})
    tree = binding.SpecTree(*([16] * 7))
    rc = lib.spec_tree_build(ctypes.byref(cfg), ctypes.c_void_p(16), ctypes.c_void_p(16),
                             ctypes.c_void_p(16), ctypes.byref(tree), ctypes.c_void_p(16), None)
    assert rc in (binding.ST_EINVAL, binding.ST_EUNSUPPORTED)


def test_null_and_misaligned_pointers_rejected(lib):
    cfg = binding.make_cfg(synth.config(1))
    tree = binding.SpecTree(*([16] * 7))
    rc = lib.spec_tree_build(ctypes.byref(cfg), None, ctypes.c_void_p(16), ctypes.c_void_p(16),
                             ctypes.byref(tree), ctypes.c_void_p(16), None)
    assert rc == binding.ST_EINVAL
    rc = lib.gdn_tree_verify(ctypes.byref(cfg), ctypes.byref(tree), *([ctypes.c_void_p(16)] * 7),
                             ctypes.c_void_p(24), None, ctypes.c_void_p(16), None)
    assert rc == binding.ST_EINVAL
    rc = lib.attn_tree_verify(ctypes.byref(cfg), None, *([ctypes.c_void_p(16)] * 8), None)
    assert rc == binding.ST_EINVAL
    rc = lib.accept_and_commit(ctypes.byref(cfg), ctypes.byref(tree), ctypes.c_void_p(16), None,
                               None, ctypes.c_void_p(16), None)
    assert rc == binding.ST_EINVAL


@pytest.mark.parametrize("temperature,reserved", [(0.0, 0), (-1.0, 0), (float("nan"), 0),
                                                  (float("inf"), 0), (1.0, 3)])
def test_sampling_parameters_rejected_before_launch(lib, temperature, reserved):
    cfg = binding.make_cfg(synth.config(7))
    tree = binding.SpecTree(*([16] * 7))
    smp = binding.SpecSampling(temperature, reserved, 1)
    p = ctypes.c_void_p(16)
    rc = lib.accept_and_commit_sampled(ctypes.byref(cfg), ctypes.byref(tree), p, ctypes.byref(smp),
                                       ctypes.byref(binding.SpecCommitIO(*([16] * 11))),
                                       ctypes.byref(binding.SpecAccept(*([16] * 4))), p, None)
    assert rc == binding.ST_EINVAL
    rc = lib.spec_verify_step_sampled(ctypes.byref(cfg), p, p, ctypes.byref(smp),
                                      ctypes.byref(tree),
                                      ctypes.byref(binding.SpecStepIO(*([16] * 5))), p,
                                      ctypes.byref(binding.SpecCommitIO(*([16] * 11))),
                                      ctypes.byref(binding.SpecAccept(*([16] * 4))), p, None)
    assert rc == binding.ST_EINVAL
    assert lib.accept_and_commit_sampled(ctypes.byref(cfg), ctypes.byref(tree), p, None,
                                         ctypes.byref(binding.SpecCommitIO(*([16] * 11))),
                                         ctypes.byref(binding.SpecAccept(*([16] * 4))), p,
                                         None) == binding.ST_EINVAL


def test_persistent_step_shapes_and_launches(lib):
    assert binding.spec_step_launches_persistent(binding.make_cfg(synth.config(1))) == 4
    assert binding.spec_step_launches_persistent(binding.make_cfg(synth.config(4))) == 1 + 32 + 1
    for bad in (synth.config(0), synth.config(2), synth.config(1).replace(n_gdn=0)):
        cfg = binding.make_cfg(bad)                # fp32 / T > 32 / no GDN layer
        assert lib.spec_step_launches_persistent(ctypes.byref(cfg)) == -1
        p = ctypes.c_void_p(16)
        rc = lib.spec_verify_step_persistent(ctypes.byref(cfg), p, p,
                                             ctypes.byref(binding.SpecTree(*([16] * 7))),
                                             ctypes.byref(binding.SpecStepIO(*([16] * 5))), p,
                                             ctypes.byref(binding.SpecCommitIO(*([16] * 11))),
                                             ctypes.byref(binding.SpecAccept(*([16] * 4))), p,
                                             None)
        assert rc == binding.ST_EUNSUPPORTED


def test_bad_io_dtype_same_code_on_both_attention_entry_points(lib):
    """An unsupported io_dtype is refused on the host, with the same code by
    the workspace call and the no-allocation call (nothing reaches a device)."""
    cfg = binding.make_cfg(synth.config(1), io_dtype=7)
    tree = binding.SpecTree(*([16] * 7))
    p = ctypes.c_void_p(16)
    rc = lib.attn_tree_verify(ctypes.byref(cfg), ctypes.byref(tree), *([p] * 8), None)
    assert rc == binding.ST_EUNSUPPORTED
    rc = lib.attn_tree_verify_noalloc(ctypes.byref(cfg), ctypes.byref(tree), *([p] * 7), None,
                                      None)
    assert rc == binding.ST_EUNSUPPORTED
    # a NULL tree is ST_EINVAL on both
    good = binding.make_cfg(synth.config(1))
    assert lib.attn_tree_verify(ctypes.byref(good), None, *([p] * 8), None) == binding.ST_EINVAL
    assert lib.attn_tree_verify_noalloc(ctypes.byref(good), None, *([p] * 7), None,
                                        None) == binding.ST_EINVAL
