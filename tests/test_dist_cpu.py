"""Multi-process (N > 1) host logic of bench.py on CPU with the gloo backend.

Rows are independent, so N GPUs run N independent replicas (weak scaling);
the only cross-rank step is the max of the timed region.  These tests run
that reduction, the aggregate-throughput arithmetic and the reference arm's
rank handling as world_size-2 process groups on 127.0.0.1, with no GPU.
"""
from __future__ import annotations

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


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        elapsed = [0.25, 0.75][rank]
        got = bench.max_over_ranks(elapsed)
        q.put((rank, got, bench.replica_seed(7, rank)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_replica_seeds_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [0.75, 0.75]      # every rank sees the slowest rank
    assert out[0][2] != out[1][2]                   # replicas draw different batches


def test_whole_job_throughput_is_aggregate_over_replicas():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_gbs(1, 50_364_416, 1000, 0.01)
    two = bench.whole_job_gbs(2, 50_364_416, 1000, 0.01)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(50_364_416 * 1000 / 0.01 / 1e9)
    assert bench.max_over_ranks(1.5) == 1.5          # not distributed: identity


def test_reference_arm_prints_once_under_torchrun_world2():
    # rank 0 times the CPU oracle and prints one JSON line; rank 1 exits 0
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "3", "--warmup", "3", "--config", "tiny_64x768_fp32"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 3 and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
