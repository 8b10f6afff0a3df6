"""The N > 1 benchmark path (replicas, one per GPU) on CPU with world size 2 over gloo.

The data path has no collective: each replica runs the whole workload on its own GPU.  What
crosses ranks is the timing: every rank's timed region is reduced with MAX and the whole-job
throughput counts all replicas' tokens over the slowest one.  These tests run that host logic
in two gloo processes, and the reference arm under torchrun (rank 0 prints, rank 1 exits 0).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [10.0 + 3 * rank, 20.0 - 5 * rank, 7.5]          # per-rank timed regions (ms)
        got = bench.reduce_max(local, world, "cpu")
        value = bench.replica_throughput(480, 50, world, got[0])
        out.put((rank, got, value))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [13.0, 20.0, 7.5]                        # every rank sees the slowest replica
        assert value == pytest.approx(480 * 50 * 2 / 13.0e-3)  # all replicas' tokens / max time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max([1.0, 2.0], 1) == [1.0, 2.0]
    assert bench.replica_throughput(10, 4, 1, 2.0) == pytest.approx(20000.0)


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "c1", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
