"""Run the CPU oracle's independent pieces on all host cores (TEST
INFRASTRUCTURE ONLY: the CPU-baseline legs of bench.py use it).

The oracle's GDN outputs, attention outputs and GDN commits are independent
across (layer, request, head): every GDN v-head and every attention kv-head
group reads only its own slice of the inputs.  These helpers run the oracle's
own functions on one such slice in a worker process, so a whole verify step
can be spread over the host's cores.  No arithmetic lives here: each helper
slices its arguments, calls the oracle, and returns the oracle's result.

The step's inputs go to every worker once, when the pool starts (they stay
resident, as they do on the GPU); a step then sends only slice indices and
the tree or acceptance of the request.  Workers are started with the "spawn"
method (a process forked after the CUDA context exists would hang).
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os
import time

import oracle

_INP = None                 # the step's inputs, resident in each worker


def _init(payload):
    global _INP
    _INP = payload
    oracle._load()
    oracle._np(payload["kv_len"])      # the marshalling's imports, before any timing


def _ping(_=None) -> int:
    return os.getpid()


def _gdn(l, b, j, i, tree_b):
    lay = _INP["gdn"][l]
    return oracle.gdn_tree(tree_b, lay["h0"][b:b + 1, j:j + 1], lay["q"][b:b + 1, :, i:i + 1],
                           lay["k"][b:b + 1, :, i:i + 1], lay["v"][b:b + 1, :, j:j + 1],
                           lay["alpha"][b:b + 1, :, j:j + 1], lay["beta"][b:b + 1, :, j:j + 1])


def _gdn_commit(l, b, j, i, acc_b):
    lay = _INP["gdn"][l]
    return oracle.commit_gdn(acc_b, lay["h0"][b:b + 1, j:j + 1], lay["k"][b:b + 1, :, i:i + 1],
                             lay["v"][b:b + 1, :, j:j + 1], lay["alpha"][b:b + 1, :, j:j + 1],
                             lay["beta"][b:b + 1, :, j:j + 1])


def _attn(l, b, g, G, tree_b):
    lay = _INP["attn"][l]
    return oracle.attn_tree(tree_b, lay["q"][b:b + 1, :, g * G:(g + 1) * G],
                            lay["k_tree"][b:b + 1, :, g:g + 1], lay["v_tree"][b:b + 1, :, g:g + 1],
                            lay["k_cache"][b:b + 1, :, g:g + 1], lay["v_cache"][b:b + 1, :, g:g + 1],
                            _INP["kv_len"][b:b + 1])


def make_pool(inp: dict, cores: int | None = None) -> cf.ProcessPoolExecutor:
    """A spawned pool whose workers hold the step's layer inputs (numpy; bf16
    as raw uint16 bits)."""
    cores = cores or os.cpu_count() or 1
    payload = {"gdn": [{k: oracle._np(v) for k, v in lay.items()} for lay in inp["gdn"]],
               "attn": [{k: oracle._np(v) for k, v in lay.items()} for lay in inp["attn"]],
               "kv_len": oracle._np(inp["kv_len"])}
    ex = cf.ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn"),
                                initializer=_init, initargs=(payload,))
    list(ex.map(_ping, range(4 * cores)))
    return ex


def verify_step(ex: cf.ProcessPoolExecutor, scfg, inp: dict, tree_fn, rows_fn) -> float:
    """One whole oracle verify step with its per-head work spread over `ex`
    (whose workers hold `inp`'s layers); returns its wall time (s).
    tree_fn(inp) builds the tree, rows_fn(inp, tree) gives the target's token
    at every row (the oracle's argmax or draw)."""
    t0 = time.perf_counter()
    tree = tree_fn(inp)
    B, G = scfg.B, scfg.Hq // scfg.Hkv
    grp = scfg.Hv // scfg.Hk
    futs = []
    for b in range(B):
        tb = {kk: vv[b:b + 1] for kk, vv in tree.items()}
        for l in range(len(inp["gdn"])):
            futs += [ex.submit(_gdn, l, b, j, j // grp, tb) for j in range(scfg.Hv)]
        for l in range(len(inp["attn"])):
            futs += [ex.submit(_attn, l, b, g, G, tb) for g in range(scfg.Hkv)]
    acc = oracle.accept(tree, rows_fn(inp, tree), scfg.m)     # meanwhile, in this process
    for f in futs:
        f.result()
    futs = []
    for b in range(B):
        ab = {kk: vv[b:b + 1] for kk, vv in acc.items()}
        for l in range(len(inp["gdn"])):
            futs += [ex.submit(_gdn_commit, l, b, j, j // grp, ab) for j in range(scfg.Hv)]
    for lay in inp["attn"]:
        oracle.commit_kv(acc, lay["k_tree"], lay["v_tree"], lay["k_cache"], lay["v_cache"],
                         inp["kv_len"])
    for f in futs:
        f.result()
    return time.perf_counter() - t0
