#!/usr/bin/env python3
"""Benchmark of the tree-verification step on one GB300.

A step = best-first tree build + every GDN layer's tree verify + every
attention layer's tree verify + argmax/acceptance/commit, all through the
C ABI on one stream, replayed as one CUDA graph.  The default workload is the
single-request configuration: 8x16 lattice, N = 24 drafts, one GDN layer
(16 q-k / 32 v heads of 128x128 fp32 state), one attention layer (32 q / 8 kv
heads of 128, KV length 4096), vocabulary 151936, bf16 I/O; synthetic seeded
inputs.  L2 is flushed (a 2 x L2 write) before every timed step.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from speculative_decoding_tree_best_gb300 import synth  # noqa: E402

METRIC = "tree_nodes_per_s (verify step: tree build + GDN + attention + accept/commit)"
UNIT = "nodes/s"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- bytes model

def algorithmic_bytes(s: synth.SpecConfig, mean_L: float, tau: float, rows=None) -> dict:
    """Bytes each phase must move at least once (fp32 state, io-typed rows).
    rows: mean tree rows a request keeps (T unless a shared budget trims it)."""
    e = 2 if s.io == "bf16" else 4
    T = s.T if rows is None else rows
    gdn_state = s.Hv * s.dk * s.dv * 4
    gdn_rows = T * (2 * s.Hk * s.dk * e + s.Hv * s.dv * e + 2 * s.Hv * 4 + s.Hv * s.dv * e)
    attn_kv = mean_L * s.Hkv * s.D * e * 2
    attn_rows = T * (s.Hq * s.D * e * 2 + s.Hkv * s.D * e * 2)
    per_req = dict(
        # lattice (+ a Markov head's rows: W1 of every candidate and the root,
        # W2 of every candidate) and the tree rows
        tree=s.m * s.K * 8 + T * 36 + (2 * s.m * s.K + 1) * s.markov_R * 4,
        gdn=s.n_gdn * (gdn_state + gdn_rows),
        attn=s.n_attn * (attn_kv + attn_rows),
        logits=T * s.V * e,
        commit=s.n_gdn * gdn_state + s.n_attn * tau * s.Hkv * s.D * e * 2,
    )
    out = {k: v * s.B for k, v in per_req.items()}
    out["step"] = sum(out.values())
    out["gdn_kernel"] = s.B * (gdn_state + gdn_rows)          # one layer, one launch
    out["attn_kernel"] = s.B * (attn_kv + attn_rows)          # one layer
    return out


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# step's kernels from ncu captures (one pass, caches flushed before each
# launch), keyed by workload, with the SHA-256 of the sources they were taken
# on: once a kernel's sources change, its figure is dropped (reported as null)
# until it is captured again.  "attn" is one attention layer: the split-KV
# partial launch plus its merge, as attn_tree_verify launches them (the fused
# step at one request runs the last merge inside the acceptance's launch).
_CSRC = "speculative_decoding_tree_best_gb300/csrc/"
TRAFFIC = {
    "attn": {"sources": tuple(_CSRC + f for f in ("attn_tree_tc.cu", "attn_tree.cu", "common.cuh",
                                                   "tc_util.cuh", "accept_util.cuh")),
             "sha256": "bf68d689be48eb3c4896edaffb96ca5aaba7af0f92117820e0af0d8d9f436d0d",
             "bytes": {"single": 20795010, "batched": 484539173}},
    "gdn": {"sources": tuple(_CSRC + f for f in ("gdn_state.cu", "gdn_tc_body.cuh", "tc_util.cuh",
                                                  "common.cuh")),
            "sha256": "e6aadbab45768a061c4bd888b7740d8f8ff93f3089938d37e2c585cfd570ba53",
            "bytes": {"single": 2601786, "batched": 60716288}},
    "argmax": {"sources": tuple(_CSRC + f for f in ("accept_commit.cu", "accept_util.cuh",
                                                     "common.cuh")),
               "sha256": "4b423f98cfdf98e67d765d2f27167a0738072068b9a3f60b5667c1fc7b1e6cbd",
               "bytes": {"single": 7620634, "batched": 182559153}},
    "commit": {"sources": tuple(_CSRC + f for f in ("accept_commit.cu", "accept_util.cuh",
                                                     "common.cuh")),
               "sha256": "4b423f98cfdf98e67d765d2f27167a0738072068b9a3f60b5667c1fc7b1e6cbd",
               "bytes": {"single": 2183997, "batched": 51951596}},
}


def sources_sha(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def kernel_traffic(kernel: str, workload: str):
    t = TRAFFIC[kernel]
    if t["sha256"] is None or sources_sha(t["sources"]) != t["sha256"]:
        return None
    return t["bytes"].get(workload)


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------- clocks (read only)

class ClockSampler:
    """Samples SM clock, power and clock-event reasons through NVML (read-only
    queries) in a background thread; falls back to nvidia-smi."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev_index: int):
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._nvml = None
        self._proc = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError
            h = ctypes.c_void_p()
            uuid = None
            try:
                uuid = "GPU-" + str(torch.cuda.get_device_properties(dev_index).uuid)
            except Exception:
                pass
            ok = uuid and nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(dev_index, ctypes.byref(h)) != 0:
                raise OSError
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._h = nv, h
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self._reasons_fn = fn or nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except OSError:
            self._nvml = None

    def _loop(self):
        nv, h = self._nvml, self._h
        mhz, r, mw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                self._reasons_fn(h, ctypes.byref(r))
                nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
                self.samples.append((mhz.value, int(r.value), mw.value / 1000.0))
            time.sleep(0.002)

    def start(self):
        if self._nvml is not None:
            self._t = threading.Thread(target=self._loop, daemon=True)
            self._t.start()
        else:
            q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active")
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(dev_index_env())], stdout=subprocess.PIPE, text=True)

    def stop(self) -> dict:
        if self._nvml is not None:
            self._stop.set()
            self._t.join()
        elif self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate()
            for line in out.strip().splitlines():
                try:
                    sm, mx, pw, rs = [x.strip() for x in line.split(",")]
                    self.samples.append((int(sm), int(rs, 16), float(pw)))
                    self.max_mhz = int(mx)
                except ValueError:
                    pass
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        reasons = 0
        for _, r, _ in self.samples:
            reasons |= r
        # samples under load: power well above the least seen (the GPU's idle draw)
        p_min = min(s[2] for s in self.samples)
        loaded = [s for s in self.samples if s[2] >= p_min + 50.0]
        return {"sm_mhz": statistics.median(s[0] for s in (loaded or self.samples)),
                "sm_mhz_all_samples": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in self.REASONS.items() if reasons & b],
                "power_w_max": max(s[2] for s in self.samples),
                "samples": len(self.samples), "samples_under_load": len(loaded),
                "window": "every timed leg of this run (steps, phases, launches, end to end)"}


def dev_index_env() -> int:
    v = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    try:
        return int(v.split(",")[int(os.environ.get("LOCAL_RANK", "0"))])
    except (ValueError, IndexError):
        return int(os.environ.get("LOCAL_RANK", "0"))


# ----------------------------------------------------------------- distributed (timing only)

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job(nodes_local: float, ms_local: float, world: int):
    """(nodes of all ranks, slowest rank's ms per step, whole-job nodes/s)."""
    nodes = sum_over_ranks(nodes_local, world)
    ms = max_over_ranks(ms_local, world)
    return nodes, ms, nodes / (ms * 1e-3)


# ----------------------------------------------------------------- CPU oracle timing

def oracle_tree(scfg, inp):
    import oracle
    if scfg.markov_R > 0:
        return oracle.tree_build_markov(inp["lat_tok"], inp["lat_base"], inp["W1"], inp["W2"],
                                        inp["root_tok"], scfg.N)
    if scfg.ragged:
        return oracle.tree_build_ragged(inp["lat_tok"], inp["lat_score"], inp["root_tok"], scfg.N,
                                        inp["m_req"], scfg.budget)
    return oracle.tree_build(inp["lat_tok"], inp["lat_score"], inp["root_tok"], scfg.N)


def oracle_rows(scfg, inp, tree):
    """The target's token at every row: the argmax, or at temperature > 0 the draw."""
    import oracle
    if scfg.temperature > 0:
        return oracle.sample_rows(inp["logits"], tree["n_nodes"], inp["kv_len"],
                                  scfg.temperature, scfg.sample_seed)[0]
    return oracle.argmax(inp["logits"])[0]


def oracle_step(scfg, inp):
    """One whole verify step of the CPU oracle, in this process."""
    import oracle
    tree = oracle_tree(scfg, inp)
    for lay in inp["gdn"]:
        oracle.gdn_tree(tree, lay["h0"], lay["q"], lay["k"], lay["v"], lay["alpha"], lay["beta"])
    for lay in inp["attn"]:
        oracle.attn_tree(tree, lay["q"], lay["k_tree"], lay["v_tree"], lay["k_cache"],
                         lay["v_cache"], inp["kv_len"])
    acc = oracle.accept(tree, oracle_rows(scfg, inp, tree), scfg.m)
    for lay in inp["gdn"]:
        oracle.commit_gdn(acc, lay["h0"], lay["k"], lay["v"], lay["alpha"], lay["beta"])
    for lay in inp["attn"]:
        oracle.commit_kv(acc, lay["k_tree"], lay["v_tree"], lay["k_cache"], lay["v_cache"],
                         inp["kv_len"])
    return tree, acc


def planted_inputs_cpu(scfg, seed):
    import oracle
    inp = synth.make_step_inputs(scfg, seed)
    tree = oracle_tree(scfg, inp)
    fc = (synth.first_child_tokens(tree["node_parent"], tree["node_rank"], tree["node_tok"],
                                   tree["n_nodes"]) if scfg.markov_R > 0 else None)
    synth.plant_logits(inp["logits"], inp["lat_tok"], inp["lat_score"], tree["node_depth"],
                       tree["n_nodes"], scfg.p_plant, inp["plant_gen"], first_child=fc,
                       gap=scfg.plant_gap)
    return inp


def oracle_pool_steps(scfg, inp, n_steps, budget_s, pool=None):
    """Whole oracle verify steps with the per-(layer, request, head) work spread
    over every host core (oracle.pool, spawned workers holding the step's
    inputs); returns (per-step seconds, cores)."""
    from oracle import pool as opool
    own = pool is None
    ex = opool.make_pool(inp) if own else pool
    cores = ex._max_workers
    times = []
    t_all = time.perf_counter()
    try:
        while len(times) < n_steps and (time.perf_counter() - t_all) < budget_s:
            times.append(opool.verify_step(ex, scfg, inp, lambda i: oracle_tree(scfg, i),
                                           lambda i, t: oracle_rows(scfg, i, t)))
    finally:
        if own:
            ex.shutdown()
    return times, cores


def cpu_baseline(scfg, inp, budget_s=12.0, max_steps=4):
    """The oracle as it stands, timed on the host cores on whole verify steps:
    on every core (the oracle's per-head calls spread over a process pool) and
    on one core.  Stacks of many layers, whose single-core oracle step runs
    for minutes, get the all-core timing only.  inp: the step's inputs with the
    planted logits."""
    from oracle import pool as opool
    ex = opool.make_pool(inp)
    try:
        oracle_pool_steps(scfg, inp, 1, budget_s, ex)          # warm-up step
        times, cores = oracle_pool_steps(scfg, inp, max_steps, budget_s, ex)
    finally:
        ex.shutdown()
    per = statistics.median(times)
    out = {"value": scfg.B * scfg.N / per, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": (f"{len(times)} whole verify steps of the C oracle (float64) on the "
                      f"'{scfg.name}' workload, its GDN/attention/commit work per (layer, "
                      f"request, head) spread over {cores} host processes, median "
                      f"{per:.3f} s/step")}
    if scfg.n_gdn + scfg.n_attn <= 2:
        one = []
        t_all = time.perf_counter()
        while len(one) < max_steps and (time.perf_counter() - t_all) < budget_s:
            t0 = time.perf_counter()
            oracle_step(scfg, inp)
            one.append(time.perf_counter() - t0)
        p1 = statistics.median(one)
        out["single_core"] = {"value": scfg.B * scfg.N / p1, "cores": 1,
                              "sample": f"{len(one)} whole steps on one core, median {p1:.3f} s"}
    return out


# ----------------------------------------------------------------- workload naming

def workload_str(scfg) -> str:
    return (f"{scfg.name}: B={scfg.B} lattice {scfg.m}x{scfg.K} N={scfg.N} "
            + (f"positions/request {'/'.join(map(str, scfg.m_cycle))} "
               f"shared budget {scfg.budget} drafts " if scfg.ragged else "")
            + (f"Markov head rank {scfg.markov_R} " if scfg.markov_R else "")
            + (f"sampled acceptance temperature {scfg.temperature:g} "
               if scfg.temperature > 0 else "")
            + f"GDN {scfg.n_gdn}x({scfg.Hk}qk/{scfg.Hv}v heads {scfg.dk}x{scfg.dv}) "
            f"attn {scfg.n_attn}x({scfg.Hq}q/{scfg.Hkv}kv heads D={scfg.D}) "
            f"KV={scfg.L}{f' (U[{scfg.L_lo},{scfg.L}] per request)' if scfg.L_lo else ''} "
            f"V={scfg.V} {scfg.io}")


# ----------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, on whole verify steps of
    the same workload, its per-head work spread over the host cores.  Under
    torchrun only rank 0 works and prints; the other ranks return at once."""
    if rank != 0:
        return
    scfg = synth.config(args.config)
    inp = planted_inputs_cpu(scfg, args.seed)
    from oracle import pool as opool
    ex = opool.make_pool(inp)
    try:
        oracle_pool_steps(scfg, inp, args.warmup, 1e9, ex)
        times, cores = oracle_pool_steps(scfg, inp, args.steps, 1e9, ex)
    finally:
        ex.shutdown()
    per = statistics.median(times)
    mean = sum(times) / len(times)
    value = scfg.B * scfg.N / mean
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_str(scfg), "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} whole verify steps of the C oracle "
                                       f"(float64), per-(layer, request, head) work on {cores} "
                                       f"host processes, mean {mean:.3f} s, median {per:.3f} s"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- our arm

def rotating_copies(t: torch.Tensor, R: int) -> torch.Tensor:
    """R device copies of t (stacked), for timing launches whose inputs are
    not in L2."""
    out = torch.empty((R,) + tuple(t.shape), dtype=t.dtype, device=t.device)
    out.copy_(t.unsqueeze(0).expand_as(out))
    return out


def measure(scfg, args, rank, world, dev, flush, steps, warmup, kernels=True, e2e=True):
    """Time one workload: the fused step graph (K replays, L2 flushed before
    each), each phase alone, the GDN and attention launches back to back over
    rotating inputs, and the end-to-end step with host buffers."""
    from speculative_decoding_tree_best_gb300 import binding
    from speculative_decoding_tree_best_gb300.step import VerifyStep, stack_inputs

    inp = synth.make_step_inputs(scfg, args.seed + rank)
    x = stack_inputs(inp, dev)
    st = VerifyStep(scfg, x, dev, persistent=args.persistent)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    # plant the target argmax along the tree the library builds (input synthesis)
    st.build_tree()
    torch.cuda.synchronize()
    t_np = st.tree.to_numpy()
    logits = inp["logits"].clone()
    fc = (synth.first_child_tokens(t_np["node_parent"], t_np["node_rank"], t_np["node_tok"],
                                   t_np["n_nodes"]) if scfg.markov_R > 0 else None)
    synth.plant_logits(logits, inp["lat_tok"], inp["lat_score"], t_np["node_depth"],
                       t_np["n_nodes"], scfg.p_plant, inp["plant_gen"], first_child=fc,
                       gap=scfg.plant_gap)
    x["logits"].copy_(logits.to(dev))
    inp["logits"] = logits                 # the oracle baseline reads the same planted rows
    kv0, root0 = x["kv_len"].clone(), x["root_tok"].clone()

    def reset():
        x["kv_len"].copy_(kv0)
        x["root_tok"].copy_(root0)

    # eager warm-up (sets kernel attributes), then capture the step as one graph
    for _ in range(3):
        reset()
        st.run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        st.run()
    torch.cuda.synchronize()
    for _ in range(warmup):
        flush.zero_()
        reset()
        graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K graph replays, L2 flushed before each -----------------------
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        reset()
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    barrier(world)
    per_ms = [a.elapsed_time(b) for a, b in ev]
    ms_step = sum(per_ms) / len(per_ms)
    tau = st.acc.accept_len.float().mean().item()
    kept = st.tree.n_nodes.float()                       # rows each request keeps
    res = {"st": st, "inp": inp, "ms_step": ms_step, "per_ms": per_ms, "wall": wall, "tau": tau,
           "drafts": int((kept - 1).sum().item()), "mean_rows": float(kept.mean().item()),
           "mean_L": float(kv0.float().mean().item())}

    # ---- each phase alone: one graph per phase, L2 flushed before every replay ------
    c = st.cfg

    def gdn_all():
        for l in range(c.n_gdn_layers):
            binding.gdn_tree_verify(c, st.tree, x["gdn_h0"][l], x["gdn_q"][l], x["gdn_k"][l],
                                    x["gdn_v"][l], x["gdn_alpha"][l], x["gdn_beta"][l],
                                    st.gdn_o[l], None, st.ws)

    def attn_all():
        for l in range(c.n_attn_layers):
            binding.attn_tree_verify(c, st.tree, x["attn_q"][l], x["k_tree"][l], x["v_tree"][l],
                                     x["k_cache"][l], x["v_cache"][l], x["kv_len"], st.attn_o[l],
                                     st.ws)

    def timed_graphs(fns: dict, reps: int) -> dict:
        graphs = {}
        for name, fn in fns.items():
            reset()
            pg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(pg, capture_error_mode="thread_local"):
                fn()
            graphs[name] = pg
        torch.cuda.synchronize()
        out = {k: [] for k in graphs}
        for _ in range(reps):
            for name, pg in graphs.items():
                flush.zero_()
                reset()
                a, bev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                pg.replay()
                bev.record(stream)
                torch.cuda.synchronize()
                out[name].append(a.elapsed_time(bev))
        return out

    R = max(10, min(steps, 50))
    ph = timed_graphs({"tree": st.build_tree, "gdn": gdn_all, "attn": attn_all,
                       "accept_commit": st.accept_commit}, R)
    res["phases_us"] = {k: 1e3 * statistics.median(v) for k, v in ph.items()}

    # ---- GDN and attention launches back to back over rotating inputs ---------------
    # (one layer's inputs copied R times, R x bytes > 2 x L2, so every launch
    # reads its inputs from HBM; the mean duration per launch includes the gaps
    # between consecutive launches)
    if kernels:
        byts = algorithmic_bytes(scfg, res["mean_L"], tau,
                                 rows=res["mean_rows"] if scfg.ragged else None)
        kus = {}
        if c.n_gdn_layers:
            Rg = int(min(128, max(2, -(-2 * l2 // int(byts["gdn_kernel"])))))
            g = {k: rotating_copies(x[k][0], Rg) for k in ("gdn_h0", "gdn_q", "gdn_k", "gdn_v",
                                                           "gdn_alpha", "gdn_beta")}
            go = rotating_copies(st.gdn_o[0], Rg)

            def gdn_rot():
                for r in range(Rg):
                    binding.gdn_tree_verify(c, st.tree, g["gdn_h0"][r], g["gdn_q"][r],
                                            g["gdn_k"][r], g["gdn_v"][r], g["gdn_alpha"][r],
                                            g["gdn_beta"][r], go[r], None, st.ws)
            t = timed_graphs({"gdn": gdn_rot}, 5)["gdn"]
            kus["gdn"] = 1e3 * statistics.median(t) / Rg
            kus["gdn_launches_timed"] = Rg
            del g, go
        if c.n_attn_layers:
            Ra = int(min(64, max(2, -(-2 * l2 // int(byts["attn_kernel"])))))
            a_ = {k: rotating_copies(x[k][0], Ra) for k in ("attn_q", "k_tree", "v_tree",
                                                            "k_cache", "v_cache")}
            ao = rotating_copies(st.attn_o[0], Ra)

            def attn_rot():
                for r in range(Ra):
                    binding.attn_tree_verify(c, st.tree, a_["attn_q"][r], a_["k_tree"][r],
                                             a_["v_tree"][r], a_["k_cache"][r], a_["v_cache"][r],
                                             x["kv_len"], ao[r], st.ws)
            t = timed_graphs({"attn": attn_rot}, 5)["attn"]
            kus["attn"] = 1e3 * statistics.median(t) / Ra
            kus["attn_launches_timed"] = Ra
            del a_, ao
        torch.cuda.empty_cache()
        res["kernel_us"] = kus

    # ---- end to end through the public API with host buffers ----------------------
    # step.HostStep: the step's inputs arrive from pinned host memory in four
    # pieces on a copy stream (lattice, attention rows, GDN rows, logits), each
    # phase waiting only for its piece, so the logits copy overlaps the tree,
    # attention and GDN; the accepted lengths and tokens go back to pinned host
    # memory.  Captured once as a CUDA graph; every timed step replays it.
    if e2e:
        from speculative_decoding_tree_best_gb300.step import HostStep
        hs = HostStep(st)
        reset()
        hs.capture()
        e2e_ms = []
        for i in range(warmup + steps):
            flush.zero_()
            reset()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            hs.run()
            b.record(stream)
            torch.cuda.synchronize()
            if i >= warmup:
                e2e_ms.append(a.elapsed_time(b))
        res["e2e_ms"] = max_over_ranks(sum(e2e_ms) / len(e2e_ms), world)
        res["h2d"] = hs.h2d_bytes
        res["d2h"] = hs.d2h_bytes
    return res


def summarize(scfg, res, world, peak, peak_kind):
    """The figures of one measured workload (rank 0 reports them)."""
    nodes_total, ms_step_max, value = whole_job(res["drafts"], res["ms_step"], world)
    byts = algorithmic_bytes(scfg, res["mean_L"], res["tau"],
                             rows=res["mean_rows"] if scfg.ragged else None)
    step_gbs = byts["step"] / (ms_step_max * 1e-3) / 1e9
    per_ms = res["per_ms"]
    kus = res.get("kernel_us", {})

    def roof(kernel, key):
        us = kus.get(kernel)
        single = res["phases_us"].get(kernel)
        n = {"gdn": max(scfg.n_gdn, 1), "attn": max(scfg.n_attn, 1)}[kernel]
        out = {"bound": "hbm", "peak": peak, "unit": "GB/s",
               "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
               if peak_kind == "measured" else "fallback",
               "algorithmic_bytes": byts[key], "traffic": kernel_traffic(kernel, scfg.name)}
        if us:
            ach = byts[key] / (us * 1e-6) / 1e9
            out.update({"achieved": ach, "frac": ach / peak, "launch_us": us,
                        "timing": f"mean of {kus[kernel + '_launches_timed']} back-to-back "
                                  "launches over rotating inputs (> 2 x L2), CUDA events"})
        if single:
            ach1 = byts[key] / (single / n * 1e-6) / 1e9
            out["single_launch"] = {"us": single / n, "achieved": ach1, "frac": ach1 / peak,
                                    "timing": "one launch per graph after an L2 flush, "
                                              "graph launch latency included"}
        return out

    out = {
        "workload": workload_str(scfg),
        "verify_step_us": ms_step_max * 1e3,
        "verify_step_us_median_p10_p90": [1e3 * statistics.median(per_ms),
                                          1e3 * sorted(per_ms)[len(per_ms) // 10],
                                          1e3 * sorted(per_ms)[(9 * len(per_ms)) // 10]],
        "tree_nodes_per_s": value,
        "step_hbm_gbs": step_gbs,
        "step_roofline_frac": step_gbs / peak,
        "step_frac_of_nominal_8tbs": step_gbs / 8000.0,
        "phases_us": res["phases_us"],
        "kernel_us": {k: v for k, v in kus.items() if not k.endswith("_timed")},
        "tau_mean": res["tau"],
        "roofline": dict(kernel="attn_tree_verify (split-KV partial + merge)", **roof("attn", "attn_kernel")),
        "gdn_roofline": dict(kernel="gdn_tree_verify", **roof("gdn", "gdn_kernel")),
        "algorithmic_bytes": byts,
        "dram_traffic_per_launch": {k: kernel_traffic(k, scfg.name) for k in TRAFFIC},
    }
    if "e2e_ms" in res:
        out["e2e"] = {"value": nodes_total / (res["e2e_ms"] * 1e-3), "unit": UNIT,
                      "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                      "ms_per_step": res["e2e_ms"]}
    return out, value, ms_step_max


def run_ours(args, rank, world, local):
    from speculative_decoding_tree_best_gb300 import binding, build

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    binding.load()
    scfg = synth.config(args.config)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    peak, peak_kind = hbm_peak()

    clocks = ClockSampler(local)
    clocks.start()                          # every leg below runs under the sampler
    res = measure(scfg, args, rank, world, dev, flush, args.steps, args.warmup)
    head, value, ms_step_max = summarize(scfg, res, world, peak, peak_kind)
    batched = None
    if args.config == 1 and not args.no_batched:
        b_cfg = synth.config(3)
        res_b = measure(b_cfg, args, rank, world, dev, flush, args.steps, args.warmup)
        batched, _, _ = summarize(b_cfg, res_b, world, peak, peak_kind)
        batched["gpu_launches"] = res_b["st"].launches_per_step * args.steps
        del res_b
    clk = clocks.stop()
    st = res["st"]
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if scfg.io == "bf16" else "f32",
        "data": "synthetic (seeded; shapes and value distributions of the paper's workloads)",
        "config": {"workload": workload_str(scfg),
                   "l2": "flushed before every timed step (2 x L2 write)",
                   "launch": "one CUDA graph per step"
                             + (", argmax/accept/GDN verify+commit in one persistent launch"
                                if args.persistent else ""),
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
    }
    line.update(head)
    line.pop("workload")
    line["clocks"] = clk
    line["gpu_launches"] = st.launches_per_step * args.steps
    line["wall_s_timed_region"] = res["wall"]
    if batched is not None:
        line["batched"] = batched
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(scfg, res["inp"])
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=1, help="workload index (see synth.CONFIGS)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-batched", action="store_true",
                    help="skip the batched (24-request) leg the default single-request run adds")
    ap.add_argument("--persistent", action="store_true",
                    help="argmax, acceptance and every GDN layer's verify + commit in one "
                         "persistent launch (spec_verify_step_persistent)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
