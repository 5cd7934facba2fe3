"""Multi-rank host logic of bench.py on CPU with gloo, world size 2.

The path needs no exchange between GPUs (independent replicas); what ranks
share is the timing reduction: the slowest rank's time and the whole-job
throughput computed from it."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        slowest = bench.reduce_max(10.0 + 5.0 * rank, world, "cpu")
        out[rank] = (slowest, bench.job_throughput(1000, 4, slowest, world))
    finally:
        dist.destroy_process_group()


def test_reduce_max_and_throughput_gloo():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 ranks x 1000 units x 4 steps in the slowest rank's 15 ms
    assert res[0][1] == pytest.approx(2 * 1000 * 4 / 0.015)


def test_single_rank_helpers():
    assert bench.reduce_max(3.5, 1, "cpu") == 3.5
    assert bench.job_throughput(647170, 30, 7.5, 1) == pytest.approx(647170 * 30 / 0.0075)


def test_reference_arm_under_torchrun_rank0_only():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--config", "tiny"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
