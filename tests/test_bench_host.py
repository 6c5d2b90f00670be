"""Host-side checks of bench.py: the multi-rank aggregation (world size 2 over
gloo on CPU) and the reference arm (the CPU oracle)."""

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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench._barrier(world)
        m = bench._max_over_ranks(times[rank], world)
        out[rank] = m
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    times = [12.5, 17.25]
    mp.start_processes(_worker, args=(2, _free_port(), times, out), nprocs=2, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == 17.25


def test_whole_job_rate_counts_all_replicas_at_the_slowest_time():
    # 2 replicas, 1e9 B per step each, 10 steps, slowest rank 2 ms total
    assert bench.whole_job_rate(1e9, 10, 2.0, 2) == pytest.approx(1e13)
    assert bench.whole_job_rate(64, 100, 10.0, 1) == pytest.approx(640000.0)


def test_reference_arm_runs_the_oracle():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
           "--steps", "2", "--warmup", "3", "--ref-seconds", "5"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["metric"] == bench.METRIC
