"""The multi-GPU path is N independent replicas (one per rank, no data-path
collective); these tests cover its host logic with world size 2 on gloo, on CPU:
the max over ranks that times the job, the job throughput, and the reference arm
launched under torchrun (rank 0 prints the only line, rank 1 exits cleanly)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank)      # rank 1 is the slow one
        out[rank] = (ms, bench.job_tflops(2e12, world, ms))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank():
    world, port = 2, free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, tf = out[r]
        assert ms == 15.0
        assert tf == pytest.approx(2 * 2e12 / 15e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(1e12, 1, 1000.0) == pytest.approx(1.0)


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--workload", "fwd_b1_h1_n128_d64", "--steps", "2",
           "--warmup", "1", "--gpus", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
