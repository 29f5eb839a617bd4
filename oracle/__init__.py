"""CPU oracle for the tree-verification step (TEST INFRASTRUCTURE ONLY).

This package is the slow, plain definition of what the CUDA library computes:
a best-first draft tree over a drafter lattice, Gated-DeltaNet outputs
recomputed along every node's root path, tree-ancestor-masked attention,
vocabulary argmax, greedy acceptance and the commit of the accepted path.  The
arithmetic lives in ``spec_oracle.c`` (plain C, float64 accumulation, built
with gcc); this module only marshals numpy/torch-CPU arrays through ctypes.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA path and never
touches a GPU.

Every function cites the section of the paper digest "SpecPilot: Autonomous
Algorithm Discovery and Systems Optimization for Speculative Decoding"
(rainbus.top) it follows; the C source holds the full statement.

Parity pins: every function here is pinned by tests under ``tests/``
(brute-force tree enumeration, closed forms, an independent ancestor-expansion
GDN formulation, float64 SDPA, torch.argmax, a plain chain verifier and the
multi-step decode consistency check; for stochastic acceptance, Philox's
published known answers and an independent implementation, chi-square tests
of the draws against the tempered softmax, and the exact law of the
speculative-decoding tutorial's rejection rule).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libspec_oracle.so")
_lock = threading.Lock()
_lib = None

ANC_WORDS = 2
MAX_ROWS = 128


def build(force: bool = False) -> str:
    """Compile spec_oracle.c with gcc (-O2, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = ctypes.CDLL(path)
            for name in ("orc_tree_build", "orc_tree_build_ragged", "orc_tree_build_markov",
                         "orc_markov_edges", "orc_exp32_log32", "orc_gdn_tree",
                         "orc_attn_tree", "orc_argmax", "orc_accept", "orc_commit_gdn",
                         "orc_commit_kv", "orc_philox4x32_10", "orc_sample_rows",
                         "orc_sample_gaps"):
                getattr(lib, name).restype = ctypes.c_int
            lib.orc_sample_rows.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p, ctypes.c_int] + \
                [ctypes.c_void_p] * 2 + [ctypes.c_double, ctypes.c_uint64, ctypes.c_int] + \
                [ctypes.c_void_p] * 2
            lib.orc_sample_gaps.argtypes = [ctypes.c_int, ctypes.c_void_p] + [ctypes.c_int] * 4 + \
                [ctypes.c_double, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
            _lib = lib
    return _lib


# ---------------------------------------------------------------- marshalling

def _np(x, dtype=None):
    """torch CPU tensor or numpy array -> contiguous numpy array.

    bf16 tensors become their raw uint16 bits (the C side widens them exactly).
    """
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16).numpy().view(np.uint16)
            else:
                x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if dtype is not None and x.dtype != dtype:
        x = np.ascontiguousarray(x.astype(dtype))
    return x


def _io(x):
    """Array of model values -> (contiguous array, io_bf16 flag)."""
    a = _np(x)
    if a.dtype == np.uint16:
        return a, 1
    return np.ascontiguousarray(a, dtype=np.float32), 0


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its input (code {rc})")


# --------------------------------------------------------------- the oracle

def tree_build(lat_tok, lat_score, root_tok, N: int) -> dict:
    """Best-first draft tree over the drafter lattice.

    Digest sections: prerequisites / draft-tree verification (nodes added
    greedily by root-path log-prob up to N) and technical novelty, Figure 6
    (best-first tree, edges scored log p(child|parent)).
    lat_tok int32 [B][m][K], lat_score f32 [B][m][K], root_tok int32 [B].
    """
    tok = _np(lat_tok, np.int32)
    sc = _np(lat_score, np.float32)
    root = _np(root_tok, np.int32).reshape(-1)
    B, m, K = tok.shape
    T = N + 1
    out = dict(
        node_tok=np.empty((B, T), np.int32), node_parent=np.empty((B, T), np.int32),
        node_depth=np.empty((B, T), np.int32), node_rank=np.empty((B, T), np.int32),
        node_score=np.empty((B, T), np.float32),
        node_anc=np.empty((B, T, ANC_WORDS), np.uint64), n_nodes=np.empty((B,), np.int32))
    rc = _load().orc_tree_build(
        B, m, K, N, _p(tok), _p(sc), _p(root), _p(out["node_tok"]), _p(out["node_parent"]),
        _p(out["node_depth"]), _p(out["node_rank"]), _p(out["node_score"]), _p(out["node_anc"]),
        _p(out["n_nodes"]))
    _check(rc, "tree_build")
    return out


def tree_build_ragged(lat_tok, lat_score, root_tok, N: int, m_req, budget: int) -> dict:
    """Best-first draft trees of a batch sharing a node budget.

    Digest section: technical novelty, batching (a node budget shared by the
    batch at the target GEMM's 192-node plateau; 16/12/8 draft positions
    chosen per request), with the tree rules of tree_build.  Request b drafts
    from its first m_req[b] lattice positions; draft nodes are inserted
    best-first over all requests' frontiers together (score desc, request asc,
    then depth, parent, rank), at most N per request, at most `budget` in all
    (budget < 0: no shared budget).
    """
    tok = _np(lat_tok, np.int32)
    sc = _np(lat_score, np.float32)
    root = _np(root_tok, np.int32).reshape(-1)
    mr = _np(m_req, np.int32).reshape(-1)
    B, m, K = tok.shape
    T = N + 1
    out = dict(
        node_tok=np.empty((B, T), np.int32), node_parent=np.empty((B, T), np.int32),
        node_depth=np.empty((B, T), np.int32), node_rank=np.empty((B, T), np.int32),
        node_score=np.empty((B, T), np.float32),
        node_anc=np.empty((B, T, ANC_WORDS), np.uint64), n_nodes=np.empty((B,), np.int32))
    rc = _load().orc_tree_build_ragged(
        B, m, K, N, _p(mr), int(budget), _p(tok), _p(sc), _p(root), _p(out["node_tok"]),
        _p(out["node_parent"]), _p(out["node_depth"]), _p(out["node_rank"]),
        _p(out["node_score"]), _p(out["node_anc"]), _p(out["n_nodes"]))
    _check(rc, "tree_build_ragged")
    return out


def exp32_log32(x, z):
    """The fp32 exp (x <= 0) and log (z >= 1) that fix the Markov edge scores to
    the bit (Cody-Waite reduction + Taylor polynomial; exponent split + atanh
    series).  Returns (exp32(x), log32(z)) as float32 arrays."""
    xa = np.ascontiguousarray(x, np.float32).reshape(-1)
    za = np.ascontiguousarray(z, np.float32).reshape(-1)
    assert xa.size == za.size
    ex = np.empty_like(xa)
    lz = np.empty_like(za)
    _check(_load().orc_exp32_log32(xa.size, _p(xa), _p(ex), _p(za), _p(lz)), "exp32_log32")
    return ex, lz


def markov_edges(x: int, tok, base, W1, W2) -> np.ndarray:
    """Edge scores of one lattice position's K candidates under a parent with
    token x: l = base + <W1[x], W2[y]>, minus their log-sum-exp (fp32, fixed
    order).  Digest section: prerequisites / parallel drafter (DSpark's Markov
    head l_s(y) = bases(y) + <W1[x_{s-1}], W2[y]>) and technical novelty (edges
    scored log p(child | parent))."""
    t = _np(tok, np.int32).reshape(-1)
    bs = _np(base, np.float32).reshape(-1)
    w1 = _np(W1, np.float32)
    w2 = _np(W2, np.float32)
    out = np.empty(t.size, np.float32)
    _check(_load().orc_markov_edges(t.size, w1.shape[1], int(x), _p(t), _p(bs), _p(w1), _p(w2),
                                    _p(out)), "markov_edges")
    return out


def tree_build_markov(lat_tok, lat_base, W1, W2, root_tok, N: int) -> dict:
    """Best-first draft tree with parent-dependent (Markov-head) edge scores:
    node n's children are ranked by markov_edges(token of n, its position).
    Outputs as tree_build."""
    tok = _np(lat_tok, np.int32)
    bs = _np(lat_base, np.float32)
    w1 = _np(W1, np.float32)
    w2 = _np(W2, np.float32)
    root = _np(root_tok, np.int32).reshape(-1)
    B, m, K = tok.shape
    T = N + 1
    out = dict(
        node_tok=np.empty((B, T), np.int32), node_parent=np.empty((B, T), np.int32),
        node_depth=np.empty((B, T), np.int32), node_rank=np.empty((B, T), np.int32),
        node_score=np.empty((B, T), np.float32),
        node_anc=np.empty((B, T, ANC_WORDS), np.uint64), n_nodes=np.empty((B,), np.int32))
    rc = _load().orc_tree_build_markov(
        B, m, K, N, w1.shape[1], _p(tok), _p(bs), _p(w1), _p(w2), _p(root), _p(out["node_tok"]),
        _p(out["node_parent"]), _p(out["node_depth"]), _p(out["node_rank"]),
        _p(out["node_score"]), _p(out["node_anc"]), _p(out["n_nodes"]))
    _check(rc, "tree_build_markov")
    return out


def gdn_tree(tree: dict, h0, q, k, v, alpha, beta) -> np.ndarray:
    """Per-node GDN output, each node decoded along its own root path.

    Digest section: prerequisites / hybrid recurrent target (gated delta rule
    h_t = a_t (I - b_t k_t k_t^T) h_{t-1} + b_t k_t v_t^T, o_t = h_t^T q_t)
    and technical novelty (recompute along the root path, no snapshots).
    h0 [B][Hv][dk][dv] (widened to float64), q/k [B][T][Hk][dk],
    v [B][T][Hv][dv], alpha/beta f32 [B][T][Hv].  Returns float64 [B][T][Hv][dv].
    """
    h = _np(h0).astype(np.float64)
    qa, bf = _io(q)
    ka, _ = _io(k)
    va, _ = _io(v)
    al = _np(alpha, np.float32)
    be = _np(beta, np.float32)
    B, T, Hk, dk = qa.shape
    Hv, dv = va.shape[2], va.shape[3]
    par = _np(tree["node_parent"], np.int32)
    nn = _np(tree["n_nodes"], np.int32)
    o = np.empty((B, T, Hv, dv), np.float64)
    rc = _load().orc_gdn_tree(B, T, Hk, Hv, dk, dv, _p(par), _p(nn), _p(h), _p(qa), _p(ka),
                              _p(va), bf, _p(al), _p(be), _p(o))
    _check(rc, "gdn_tree")
    return o


def attn_tree(tree: dict, q, k_tree, v_tree, k_cache, v_cache, kv_len) -> np.ndarray:
    """Tree-ancestor-masked attention of every node over cache + ancestors.

    Digest section: prerequisites / draft-tree verification (each node sees
    only its ancestors).  q [B][T][Hq][D], k_tree/v_tree [B][T][Hkv][D],
    k_cache/v_cache [B][Lmax][Hkv][D], kv_len [B].  Returns float64 [B][T][Hq][D].
    """
    qa, bf = _io(q)
    kt, _ = _io(k_tree)
    vt, _ = _io(v_tree)
    kc, _ = _io(k_cache)
    vc, _ = _io(v_cache)
    L = _np(kv_len, np.int32).reshape(-1)
    B, T, Hq, D = qa.shape
    Hkv, Lmax = kt.shape[2], kc.shape[1]
    nn = _np(tree["n_nodes"], np.int32)
    anc = _np(tree["node_anc"], np.uint64)
    o = np.empty((B, T, Hq, D), np.float64)
    rc = _load().orc_attn_tree(B, T, Hq, Hkv, D, Lmax, _p(nn), _p(anc), _p(qa), _p(kt), _p(vt),
                               _p(kc), _p(vc), _p(L), bf, _p(o))
    _check(rc, "attn_tree")
    return o


def argmax(logits):
    """First-index argmax of each row and its top-2 margin.

    Digest section: prerequisites / speculative decoding (accept tokens equal
    to the target argmax).  logits [..., V]; returns (int32 [...], f32 [...]).
    """
    la, bf = _io(logits)
    V = la.shape[-1]
    lead = la.shape[:-1]
    rows = int(np.prod(lead)) if lead else 1
    idx = np.empty((rows,), np.int32)
    mar = np.empty((rows,), np.float32)
    rc = _load().orc_argmax(rows, V, _p(la), bf, _p(idx), _p(mar))
    _check(rc, "argmax")
    return idx.reshape(lead), mar.reshape(lead)


SAMPLE_CHUNK = 4096


def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox4x32-10 blocks: ctr uint32 [n][4], key uint32 [n][2] -> uint32 [n][4].

    Definition: Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy
    as 1, 2, 3" (SC 2011)."""
    c = _np(ctr, np.uint32).reshape(-1, 4)
    k = _np(key, np.uint32).reshape(-1, 2)
    assert c.shape[0] == k.shape[0]
    out = np.empty_like(c)
    _load().orc_philox4x32_10(c.shape[0], _p(c), _p(k), _p(out))
    return out


def sample_rows(logits, n_nodes, kv_len, temperature: float, seed: int,
                chunk: int = SAMPLE_CHUNK):
    """The target's draw from softmax(logits / temperature) at every tree row
    (two-level Gumbel-max, Philox4x32-10 noise keyed by seed and counted by
    (index, row, request, kv_len)).

    Speculative-decoding tutorial (mlqm.cn), section 2.3: with fixed draft
    tokens the rejection rule is the same law as following the child whose
    token equals the target's draw.  logits [B][T][V]; returns (int32 [B][T],
    float64 [B][T] margin); padding rows get -1 and +inf."""
    la, bf = _io(logits)
    B, T, V = la.shape
    nn = _np(n_nodes, np.int32)
    kl = _np(kv_len, np.int32)
    smp = np.empty((B, T), np.int32)
    mar = np.empty((B, T), np.float64)
    rc = _load().orc_sample_rows(B, T, V, _p(la), bf, _p(nn), _p(kl), float(temperature),
                                 int(seed) & 0xFFFFFFFFFFFFFFFF, int(chunk), _p(smp), _p(mar))
    _check(rc, "sample_rows")
    return smp, mar


def sample_gaps(row_logits, t: int, b: int, pos: int, temperature: float, seed: int, alt: int,
                chunk: int = SAMPLE_CHUNK):
    """How far token `alt` falls behind row (b, t)'s draw: (chunk-level gap,
    token-level gap); both 0 when alt is the draw."""
    la, bf = _io(row_logits)
    gaps = np.empty((2,), np.float64)
    rc = _load().orc_sample_gaps(la.shape[-1], _p(la), bf, int(t), int(b), int(pos),
                                 float(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF, int(chunk),
                                 int(alt), _p(gaps))
    _check(rc, "sample_gaps")
    return float(gaps[0]), float(gaps[1])


def accept(tree: dict, argmax_rows, m: int) -> dict:
    """Longest root path matching the target argmax, plus the bonus token.

    Digest sections: prerequisites / speculative decoding (tau in [1, m+1])
    and draft-tree verification (longest matching root path + bonus).
    argmax_rows int32 [B][T].
    """
    tok = _np(tree["node_tok"], np.int32)
    par = _np(tree["node_parent"], np.int32)
    nn = _np(tree["n_nodes"], np.int32)
    am = _np(argmax_rows, np.int32)
    B, T = tok.shape
    out = dict(accept_len=np.empty((B,), np.int32),
               accept_nodes=np.empty((B, m + 1), np.int32),
               out_tok=np.empty((B, m + 1), np.int32), new_root=np.empty((B,), np.int32))
    rc = _load().orc_accept(B, T, m, _p(tok), _p(par), _p(nn), _p(am), _p(out["accept_len"]),
                            _p(out["accept_nodes"]), _p(out["out_tok"]), _p(out["new_root"]))
    _check(rc, "accept")
    return out


def commit_gdn(acc: dict, h, k, v, alpha, beta) -> np.ndarray:
    """State after the accepted path's gated-delta steps (one GDN layer).

    Digest sections: hybrid recurrent target and technical novelty (the
    committed state is recomputed along the accepted root path).
    Returns a new float64 [B][Hv][dk][dv].
    """
    hh = np.array(_np(h), dtype=np.float64, copy=True)
    ka, bf = _io(k)
    va, _ = _io(v)
    al = _np(alpha, np.float32)
    be = _np(beta, np.float32)
    B, T, Hk, dk = ka.shape
    Hv, dv = va.shape[2], va.shape[3]
    alen = _np(acc["accept_len"], np.int32)
    anodes = _np(acc["accept_nodes"], np.int32)
    m = anodes.shape[1] - 1
    rc = _load().orc_commit_gdn(B, T, m, Hk, Hv, dk, dv, _p(alen), _p(anodes), _p(hh), _p(ka),
                                _p(va), bf, _p(al), _p(be))
    _check(rc, "commit_gdn")
    return hh


def commit_kv(acc: dict, k_tree, v_tree, k_cache, v_cache, kv_len):
    """Append the accepted path's tree K/V rows to the cache (one layer).

    Returns new (k_cache, v_cache) arrays in the input element type (bf16 as
    raw uint16 bits).  Raises ValueError on cache overflow.
    """
    kt, bf = _io(k_tree)
    vt, _ = _io(v_tree)
    kc = np.array(_io(k_cache)[0], copy=True)
    vc = np.array(_io(v_cache)[0], copy=True)
    B, T, Hkv, D = kt.shape
    Lmax = kc.shape[1]
    L = _np(kv_len, np.int32).reshape(-1)
    alen = _np(acc["accept_len"], np.int32)
    anodes = _np(acc["accept_nodes"], np.int32)
    m = anodes.shape[1] - 1
    rc = _load().orc_commit_kv(B, T, m, Hkv, D, Lmax, _p(alen), _p(anodes), _p(kt), _p(vt),
                               _p(kc), _p(vc), _p(L), bf)
    _check(rc, "commit_kv")
    return kc, vc
