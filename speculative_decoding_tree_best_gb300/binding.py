"""Thin ctypes binding of libspectree (include/spec_tree.h).

The functions below carry the C entry points' names and do argument
marshalling only: they check that tensors are CUDA, contiguous and of the
expected dtype, then pass raw device pointers and the current CUDA stream.
Every step of the computation runs in the library's kernels; there is no
fallback, and loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspectree.so")

ST_OK, ST_EINVAL, ST_EUNSUPPORTED, ST_ECUDA, ST_EOVERFLOW, ST_TIMEOUT, ST_ESCRATCH = range(7)
NOALLOC_SCRATCH_BYTES = 8 << 20
SPEC_DEV_OVERFLOW, SPEC_DEV_BADLAT, SPEC_DEV_TIMEOUT, SPEC_DEV_BADREQ = 0x1, 0x2, 0x4, 0x8
SPEC_DEV_BADLOGIT, SPEC_DEV_RANGE = 0x10, 0x20
SPEC_IO_F32, SPEC_IO_BF16 = 0, 1
EXPORTS = ("spec_workspace_bytes", "spec_workspace_bytes_for_sms", "spec_tree_build", "gdn_tree_verify", "attn_tree_verify",
           "accept_and_commit", "spec_verify_step", "spec_status_read", "spec_status_clear",
           "spec_status_string", "spec_abi_version", "attn_tree_verify_noalloc",
           "spec_wait_probe", "spec_step_launches", "spec_tree_build_ragged",
           "spec_verify_step_ragged", "spec_tree_build_markov", "spec_verify_step_markov",
           "accept_and_commit_sampled", "spec_verify_step_sampled",
           "spec_verify_step_persistent", "spec_step_launches_persistent")
SAMPLE_CHUNK = 4096

_lock = threading.Lock()
_lib = None


class SpecError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} returned {code}: {msg}")
        self.code = code


class SpecCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "B", "m", "K", "N", "Hk", "Hv", "dk", "dv", "Hq", "Hkv", "D", "Lmax", "V",
        "n_gdn_layers", "n_attn_layers", "io_dtype")]


class SpecTree(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "node_tok", "node_parent", "node_depth", "node_rank", "node_score", "node_anc", "n_nodes")]


class SpecCommitIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "h0", "gdn_k", "gdn_v", "alpha", "beta", "k_tree", "v_tree", "k_cache", "v_cache",
        "kv_len", "root_tok")]


class SpecStepIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gdn_q", "gdn_o", "gdn_c", "attn_q", "attn_o")]


class SpecAccept(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("argmax", "accept_len", "accept_nodes", "out_tok")]


class SpecSampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("reserved", ctypes.c_uint32),
                ("seed", ctypes.c_uint64)]


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libspectree.so (raises if it is missing: build it first)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libspectree not built ({p} missing): run "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(p)
            vp, cfgp = ctypes.c_void_p, ctypes.POINTER(SpecCfg)
            lib.spec_workspace_bytes.argtypes = [cfgp]
            lib.spec_workspace_bytes.restype = ctypes.c_size_t
            lib.spec_workspace_bytes_for_sms.argtypes = [cfgp, ctypes.c_int]
            lib.spec_workspace_bytes_for_sms.restype = ctypes.c_size_t
            lib.spec_tree_build.argtypes = [cfgp, vp, vp, vp, ctypes.POINTER(SpecTree), vp, vp]
            lib.gdn_tree_verify.argtypes = [cfgp, ctypes.POINTER(SpecTree)] + [vp] * 10
            lib.attn_tree_verify.argtypes = [cfgp, ctypes.POINTER(SpecTree)] + [vp] * 9
            lib.accept_and_commit.argtypes = [cfgp, ctypes.POINTER(SpecTree), vp,
                                              ctypes.POINTER(SpecCommitIO),
                                              ctypes.POINTER(SpecAccept), vp, vp]
            lib.spec_verify_step.argtypes = [cfgp, vp, vp, ctypes.POINTER(SpecTree),
                                             ctypes.POINTER(SpecStepIO), vp,
                                             ctypes.POINTER(SpecCommitIO),
                                             ctypes.POINTER(SpecAccept), vp, vp]
            lib.spec_tree_build_ragged.argtypes = [cfgp, vp, vp, vp, vp, ctypes.c_int,
                                                   ctypes.POINTER(SpecTree), vp, vp]
            lib.spec_verify_step_ragged.argtypes = [cfgp, vp, vp, vp, ctypes.c_int,
                                                    ctypes.POINTER(SpecTree),
                                                    ctypes.POINTER(SpecStepIO), vp,
                                                    ctypes.POINTER(SpecCommitIO),
                                                    ctypes.POINTER(SpecAccept), vp, vp]
            lib.spec_tree_build_markov.argtypes = [cfgp, vp, vp, vp, vp, ctypes.c_int, vp,
                                                   ctypes.POINTER(SpecTree), vp, vp]
            lib.spec_verify_step_markov.argtypes = [cfgp, vp, vp, vp, vp, ctypes.c_int,
                                                    ctypes.POINTER(SpecTree),
                                                    ctypes.POINTER(SpecStepIO), vp,
                                                    ctypes.POINTER(SpecCommitIO),
                                                    ctypes.POINTER(SpecAccept), vp, vp]
            smpp = ctypes.POINTER(SpecSampling)
            lib.accept_and_commit_sampled.argtypes = [cfgp, ctypes.POINTER(SpecTree), vp, smpp,
                                                      ctypes.POINTER(SpecCommitIO),
                                                      ctypes.POINTER(SpecAccept), vp, vp]
            lib.spec_verify_step_sampled.argtypes = [cfgp, vp, vp, smpp, ctypes.POINTER(SpecTree),
                                                     ctypes.POINTER(SpecStepIO), vp,
                                                     ctypes.POINTER(SpecCommitIO),
                                                     ctypes.POINTER(SpecAccept), vp, vp]
            lib.spec_verify_step_persistent.argtypes = lib.spec_verify_step.argtypes
            lib.spec_step_launches_persistent.argtypes = [cfgp]
            lib.spec_status_read.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
            lib.spec_status_clear.argtypes = [vp, vp]
            lib.spec_status_string.argtypes = [ctypes.c_int]
            lib.spec_status_string.restype = ctypes.c_char_p
            lib.attn_tree_verify_noalloc.argtypes = [cfgp, ctypes.POINTER(SpecTree)] + [vp] * 9
            lib.spec_wait_probe.argtypes = [ctypes.c_uint32, ctypes.c_int, vp, vp]
            lib.spec_step_launches.argtypes = [cfgp]
            for n in ("spec_tree_build", "gdn_tree_verify", "attn_tree_verify",
                      "attn_tree_verify_noalloc", "spec_wait_probe", "spec_step_launches",
                      "spec_tree_build_ragged", "spec_verify_step_ragged", "spec_tree_build_markov",
                      "spec_verify_step_markov", "accept_and_commit_sampled",
                      "spec_verify_step_sampled", "spec_verify_step_persistent",
                      "spec_step_launches_persistent", "accept_and_commit", "spec_verify_step", "spec_status_read",
                      "spec_status_clear", "spec_abi_version"):
                getattr(lib, n).restype = ctypes.c_int
            _lib = lib
    return _lib


# ------------------------------------------------------------------ helpers

def make_cfg(sc, **over) -> SpecCfg:
    """SpecCfg from a synth.SpecConfig (or any object with the same fields)."""
    d = dict(B=sc.B, m=sc.m, K=sc.K, N=sc.N, Hk=sc.Hk, Hv=sc.Hv, dk=sc.dk, dv=sc.dv, Hq=sc.Hq,
             Hkv=sc.Hkv, D=sc.D, Lmax=sc.Lmax, V=sc.V, n_gdn_layers=sc.n_gdn,
             n_attn_layers=sc.n_attn, io_dtype=SPEC_IO_BF16 if sc.io == "bf16" else SPEC_IO_F32)
    d.update(over)
    return SpecCfg(**d)


def _io_dtype(cfg: SpecCfg):
    return torch.bfloat16 if cfg.io_dtype == SPEC_IO_BF16 else torch.float32


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn, rc):
    if rc != ST_OK:
        raise SpecError(fn, rc, load().spec_status_string(rc).decode())


class TreeBuffers:
    """Device buffers of a spec_tree for B requests and T = N + 1 rows."""

    def __init__(self, cfg: SpecCfg, device="cuda"):
        B, T = cfg.B, cfg.N + 1
        i32 = dict(dtype=torch.int32, device=device)
        self.node_tok = torch.empty((B, T), **i32)
        self.node_parent = torch.empty((B, T), **i32)
        self.node_depth = torch.empty((B, T), **i32)
        self.node_rank = torch.empty((B, T), **i32)
        self.node_score = torch.empty((B, T), dtype=torch.float32, device=device)
        self.node_anc = torch.empty((B, T, 2), dtype=torch.int64, device=device)
        self.n_nodes = torch.empty((B,), **i32)

    def c(self) -> SpecTree:
        return SpecTree(*(t.data_ptr() for t in (
            self.node_tok, self.node_parent, self.node_depth, self.node_rank, self.node_score,
            self.node_anc, self.n_nodes)))

    def to_numpy(self) -> dict:
        import numpy as np
        d = {k: getattr(self, k).cpu().numpy() for k in (
            "node_tok", "node_parent", "node_depth", "node_rank", "node_score", "n_nodes")}
        d["node_anc"] = self.node_anc.cpu().numpy().view(np.uint64)
        return d


class AcceptBuffers:
    def __init__(self, cfg: SpecCfg, device="cuda"):
        B, T, m = cfg.B, cfg.N + 1, cfg.m
        i32 = dict(dtype=torch.int32, device=device)
        self.argmax = torch.empty((B, T), **i32)
        self.accept_len = torch.empty((B,), **i32)
        self.accept_nodes = torch.empty((B, m + 1), **i32)
        self.out_tok = torch.empty((B, m + 1), **i32)

    def c(self) -> SpecAccept:
        return SpecAccept(self.argmax.data_ptr(), self.accept_len.data_ptr(),
                          self.accept_nodes.data_ptr(), self.out_tok.data_ptr())


# ------------------------------------------------------------- entry points

def spec_workspace_bytes(cfg: SpecCfg) -> int:
    """Workspace bytes for the current device."""
    n = load().spec_workspace_bytes(ctypes.byref(cfg))
    if n == 0:
        raise SpecError("spec_workspace_bytes", ST_EINVAL,
                        "invalid configuration (or no CUDA device visible)")
    return int(n)


def spec_workspace_bytes_for_sms(cfg: SpecCfg, num_sms: int) -> int:
    """Workspace bytes for a device with num_sms SMs (host only)."""
    n = load().spec_workspace_bytes_for_sms(ctypes.byref(cfg), int(num_sms))
    if n == 0:
        raise SpecError("spec_workspace_bytes_for_sms", ST_EINVAL, "invalid configuration")
    return int(n)


def alloc_workspace(cfg: SpecCfg, device="cuda") -> torch.Tensor:
    """Zero-filled workspace of spec_workspace_bytes(cfg) bytes."""
    return torch.zeros((spec_workspace_bytes(cfg),), dtype=torch.uint8, device=device)


def spec_tree_build(cfg, lat_tok, lat_score, root_tok, tree: TreeBuffers, ws, stream=None):
    _check("spec_tree_build", load().spec_tree_build(
        ctypes.byref(cfg), _ptr(lat_tok, torch.int32, "lat_tok"),
        _ptr(lat_score, torch.float32, "lat_score"), _ptr(root_tok, torch.int32, "root_tok"),
        ctypes.byref(tree.c()), _ptr(ws, name="ws"), _stream(stream)))


def gdn_tree_verify(cfg, tree: TreeBuffers, h0, q, k, v, alpha, beta, o, c=None, ws=None,
                    stream=None):
    dt = _io_dtype(cfg)
    _check("gdn_tree_verify", load().gdn_tree_verify(
        ctypes.byref(cfg), ctypes.byref(tree.c()), _ptr(h0, torch.float32, "h0"),
        _ptr(q, dt, "q"), _ptr(k, dt, "k"), _ptr(v, dt, "v"), _ptr(alpha, torch.float32, "alpha"),
        _ptr(beta, torch.float32, "beta"), _ptr(o, dt, "o"), _ptr(c, torch.float32, "c"),
        _ptr(ws, name="ws"), _stream(stream)))


def attn_tree_verify(cfg, tree: TreeBuffers, q, k_tree, v_tree, k_cache, v_cache, kv_len, o, ws,
                     stream=None):
    dt = _io_dtype(cfg)
    _check("attn_tree_verify", load().attn_tree_verify(
        ctypes.byref(cfg), ctypes.byref(tree.c()), _ptr(q, dt, "q"), _ptr(k_tree, dt, "k_tree"),
        _ptr(v_tree, dt, "v_tree"), _ptr(k_cache, dt, "k_cache"), _ptr(v_cache, dt, "v_cache"),
        _ptr(kv_len, torch.int32, "kv_len"), _ptr(o, dt, "o"), _ptr(ws, name="ws"),
        _stream(stream)))


def attn_tree_verify_noalloc(cfg, tree: TreeBuffers, q, k_tree, v_tree, k_cache, v_cache, kv_len,
                             o, dev_status=None, stream=None):
    """attn_tree_verify with the library's static scratch (no workspace);
    dev_status: None or a CUDA uint32/int32 word that receives SPEC_DEV_* bits."""
    dt = _io_dtype(cfg)
    if dev_status is not None and dev_status.dtype not in (torch.int32, torch.uint32):
        raise TypeError("dev_status: expected an int32 or uint32 CUDA tensor")
    _check("attn_tree_verify_noalloc", load().attn_tree_verify_noalloc(
        ctypes.byref(cfg), ctypes.byref(tree.c()), _ptr(q, dt, "q"), _ptr(k_tree, dt, "k_tree"),
        _ptr(v_tree, dt, "v_tree"), _ptr(k_cache, dt, "k_cache"), _ptr(v_cache, dt, "v_cache"),
        _ptr(kv_len, torch.int32, "kv_len"), _ptr(o, dt, "o"),
        _ptr(dev_status, name="dev_status"), _stream(stream)))


def _commit_io(cfg, io: dict) -> SpecCommitIO:
    dt = _io_dtype(cfg)
    f32, i32 = torch.float32, torch.int32
    types = dict(h0=f32, gdn_k=dt, gdn_v=dt, alpha=f32, beta=f32, k_tree=dt, v_tree=dt,
                 k_cache=dt, v_cache=dt, kv_len=i32, root_tok=i32)
    return SpecCommitIO(*(_ptr(io.get(n), types[n], n) for n in types))


def accept_and_commit(cfg, tree: TreeBuffers, logits, io: dict, out: AcceptBuffers, ws,
                      stream=None):
    """io: dict with stacked h0, gdn_k, gdn_v, alpha, beta, k_tree, v_tree,
    k_cache, v_cache (None allowed where the layer count is 0), kv_len, root_tok."""
    dt = _io_dtype(cfg)
    cio = _commit_io(cfg, io)
    _check("accept_and_commit", load().accept_and_commit(
        ctypes.byref(cfg), ctypes.byref(tree.c()), _ptr(logits, dt, "logits"), ctypes.byref(cio),
        ctypes.byref(out.c()), _ptr(ws, name="ws"), _stream(stream)))


def sampling(temperature: float, seed: int) -> SpecSampling:
    return SpecSampling(float(temperature), 0, int(seed) & 0xFFFFFFFFFFFFFFFF)


def accept_and_commit_sampled(cfg, tree: TreeBuffers, logits, smp: SpecSampling, io: dict,
                              out: AcceptBuffers, ws, stream=None):
    """accept_and_commit at temperature > 0: out.argmax receives each row's draw."""
    dt = _io_dtype(cfg)
    cio = _commit_io(cfg, io)
    _check("accept_and_commit_sampled", load().accept_and_commit_sampled(
        ctypes.byref(cfg), ctypes.byref(tree.c()), _ptr(logits, dt, "logits"), ctypes.byref(smp),
        ctypes.byref(cio), ctypes.byref(out.c()), _ptr(ws, name="ws"), _stream(stream)))


def spec_tree_build_ragged(cfg, lat_tok, lat_score, root_tok, m_req, node_budget: int,
                           tree: TreeBuffers, ws, stream=None):
    """Trees with per-request draft positions (m_req: CUDA int32 [B] or None) and
    a node budget shared by the batch (node_budget < 0: none)."""
    _check("spec_tree_build_ragged", load().spec_tree_build_ragged(
        ctypes.byref(cfg), _ptr(lat_tok, torch.int32, "lat_tok"),
        _ptr(lat_score, torch.float32, "lat_score"), _ptr(root_tok, torch.int32, "root_tok"),
        _ptr(m_req, torch.int32, "m_req"), int(node_budget), ctypes.byref(tree.c()),
        _ptr(ws, name="ws"), _stream(stream)))


def spec_tree_build_markov(cfg, lat_tok, lat_base, W1, W2, root_tok, tree: TreeBuffers, ws,
                           stream=None):
    """Best-first tree with Markov-head edge scores (W1, W2: CUDA f32 [V][R])."""
    _check("spec_tree_build_markov", load().spec_tree_build_markov(
        ctypes.byref(cfg), _ptr(lat_tok, torch.int32, "lat_tok"),
        _ptr(lat_base, torch.float32, "lat_base"), _ptr(W1, torch.float32, "W1"),
        _ptr(W2, torch.float32, "W2"), int(W1.shape[1]), _ptr(root_tok, torch.int32, "root_tok"),
        ctypes.byref(tree.c()), _ptr(ws, name="ws"), _stream(stream)))


def _step_io(cfg, step: dict) -> SpecStepIO:
    dt = _io_dtype(cfg)
    return SpecStepIO(_ptr(step.get("gdn_q"), dt, "gdn_q"), _ptr(step.get("gdn_o"), dt, "gdn_o"),
                      _ptr(step.get("gdn_c"), torch.float32, "gdn_c"),
                      _ptr(step.get("attn_q"), dt, "attn_q"), _ptr(step.get("attn_o"), dt, "attn_o"))


def spec_verify_step(cfg, lat_tok, lat_score, tree: TreeBuffers, step: dict, logits, io: dict,
                     out: AcceptBuffers, ws, stream=None):
    """Whole verify step (tree, every GDN and attention layer, accept+commit).
    step: dict with stacked gdn_q, gdn_o, gdn_c (or None), attn_q, attn_o."""
    dt = _io_dtype(cfg)
    sio = _step_io(cfg, step)
    _check("spec_verify_step", load().spec_verify_step(
        ctypes.byref(cfg), _ptr(lat_tok, torch.int32, "lat_tok"),
        _ptr(lat_score, torch.float32, "lat_score"), ctypes.byref(tree.c()), ctypes.byref(sio),
        _ptr(logits, dt, "logits"), ctypes.byref(_commit_io(cfg, io)), ctypes.byref(out.c()),
        _ptr(ws, name="ws"), _stream(stream)))


def spec_verify_step_persistent(cfg, lat_tok, lat_score, tree: TreeBuffers, step: dict, logits,
                                io: dict, out: AcceptBuffers, ws, stream=None):
    """spec_verify_step with the argmax, acceptance and every GDN layer's
    verify + commit in one persistent launch."""
    dt = _io_dtype(cfg)
    sio = _step_io(cfg, step)
    _check("spec_verify_step_persistent", load().spec_verify_step_persistent(
        ctypes.byref(cfg), _ptr(lat_tok, torch.int32, "lat_tok"),
        _ptr(lat_score, torch.float32, "lat_score"), ctypes.byref(tree.c()), ctypes.byref(sio),
        _ptr(logits, dt, "logits"), ctypes.byref(_commit_io(cfg, io)), ctypes.byref(out.c()),
        _ptr(ws, name="ws"), _stream(stream)))


def spec_step_launches_persistent(cfg) -> int:
    return int(load().spec_step_launches_persistent(ctypes.byref(cfg)))


def spec_verify_step_sampled(cfg, lat_tok, lat_score, smp: SpecSampling, tree: TreeBuffers,
                             step: dict, logits, io: dict, out: AcceptBuffers, ws, stream=None):
    """spec_verify_step with the sampled acceptance."""
    dt = _io_dtype(cfg)
    sio = _step_io(cfg, step)
    _check("spec_verify_step_sampled", load().spec_verify_step_sampled(
        ctypes.byref(cfg), _ptr(lat_tok, torch.int32, "lat_tok"),
        _ptr(lat_score, torch.float32, "lat_score"), ctypes.byref(smp), ctypes.byref(tree.c()),
        ctypes.byref(sio), _ptr(logits, dt, "logits"), ctypes.byref(_commit_io(cfg, io)),
        ctypes.byref(out.c()), _ptr(ws, name="ws"), _stream(stream)))


def spec_verify_step_ragged(cfg, lat_tok, lat_score, m_req, node_budget: int, tree: TreeBuffers,
                            step: dict, logits, io: dict, out: AcceptBuffers, ws, stream=None):
    """spec_verify_step over the trees of spec_tree_build_ragged."""
    dt = _io_dtype(cfg)
    sio = _step_io(cfg, step)
    _check("spec_verify_step_ragged", load().spec_verify_step_ragged(
        ctypes.byref(cfg), _ptr(lat_tok, torch.int32, "lat_tok"),
        _ptr(lat_score, torch.float32, "lat_score"), _ptr(m_req, torch.int32, "m_req"),
        int(node_budget), ctypes.byref(tree.c()), ctypes.byref(sio), _ptr(logits, dt, "logits"),
        ctypes.byref(_commit_io(cfg, io)), ctypes.byref(out.c()), _ptr(ws, name="ws"),
        _stream(stream)))


def spec_verify_step_markov(cfg, lat_tok, lat_base, W1, W2, tree: TreeBuffers, step: dict, logits,
                            io: dict, out: AcceptBuffers, ws, stream=None):
    """spec_verify_step over the tree of spec_tree_build_markov."""
    dt = _io_dtype(cfg)
    sio = _step_io(cfg, step)
    _check("spec_verify_step_markov", load().spec_verify_step_markov(
        ctypes.byref(cfg), _ptr(lat_tok, torch.int32, "lat_tok"),
        _ptr(lat_base, torch.float32, "lat_base"), _ptr(W1, torch.float32, "W1"),
        _ptr(W2, torch.float32, "W2"), int(W1.shape[1]), ctypes.byref(tree.c()),
        ctypes.byref(sio), _ptr(logits, dt, "logits"), ctypes.byref(_commit_io(cfg, io)),
        ctypes.byref(out.c()), _ptr(ws, name="ws"), _stream(stream)))


def spec_status_read(ws, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check("spec_status_read", load().spec_status_read(_ptr(ws, name="ws"), ctypes.byref(v),
                                                       _stream(stream)))
    return int(v.value)


def spec_step_launches(cfg) -> int:
    """Kernel launches one spec_verify_step call makes (host only)."""
    n = load().spec_step_launches(ctypes.byref(cfg))
    if n < 0:
        raise SpecError("spec_step_launches", ST_EINVAL, "invalid cfg")
    return n


def spec_wait_probe(limit_us: int, satisfy: bool, ws, stream=None):
    """One bounded device wait (diagnostic): SPEC_DEV_TIMEOUT when unsatisfied."""
    _check("spec_wait_probe", load().spec_wait_probe(int(limit_us), int(bool(satisfy)),
                                                     _ptr(ws, name="ws"), _stream(stream)))


def spec_status_clear(ws, stream=None):
    _check("spec_status_clear", load().spec_status_clear(_ptr(ws, name="ws"), _stream(stream)))
