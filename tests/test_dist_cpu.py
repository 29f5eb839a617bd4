"""The N > 1 path of bench.py on the CPU (gloo, world size 2): replicas with
no data-path collective; whole-job nodes/s = nodes of all ranks / slowest
rank's time; only rank 0 prints; the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import argparse

    import torch.distributed as dist

    import bench
    args = argparse.Namespace(impl="reference")
    r, w, local = bench.dist_setup(args)
    try:
        assert (r, w, local) == (rank, world, rank)
        assert dist.get_backend() == "gloo"
        # rank r processed 24 * (r + 1) nodes in (1 + r) ms per step
        nodes, ms, value = bench.whole_job(24.0 * (rank + 1), 1.0 + rank, world)
        assert bench.max_over_ranks(float(rank), world) == world - 1
        bench.barrier(world)
        q.put((rank, nodes, ms, value))
    finally:
        dist.destroy_process_group()


def test_whole_job_aggregation_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, nodes, ms, value in res:
        assert nodes == 24.0 + 48.0 and ms == 2.0
        assert value == pytest.approx(72.0 / 2e-3)


def test_reference_arm_under_torchrun_prints_one_line():
    """torchrun with 2 ranks: rank 0 times the oracle and prints one JSON line;
    rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--config", "0", "--steps", "3",
           "--warmup", "3"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    out = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
    # the rest of the line's contract
    for k in ("metric", "unit", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config"):
        assert k in rec, k
    assert rec["steps"] == 3 and rec["warmup"] == 3 and rec["higher_is_better"] is True
    assert rec["cpu_baseline"]["cores"] >= 1 and rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["e2e"]["value"] == rec["value"] and "workload" in rec["config"]
    # the same workload string as the GPU arm's line
    import bench
    from speculative_decoding_tree_best_gb300 import synth
    assert rec["config"]["workload"] == bench.workload_str(synth.config(0))
    # whole oracle steps: the line's time per step is what the run took
    assert rec["ms_per_step"] > 0
