"""The N-GPU path of bench.py without GPUs: two gloo ranks on the CPU.

Sequences are independent, so N GPUs run N replicas with no collective in
the step; the only cross-rank work is the timing reduction (the slowest
rank's timed region, the tokens of all ranks) and rank 0 printing the line.
These tests run that reduction in two processes, and check that the
reference arm does its work on rank 0 only.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, n = bench.reduce_over_ranks(10.0 + 5.0 * rank, 7 * (rank + 1), world)
    q.put((rank, ms, n))
    dist.destroy_process_group()


def test_reduce_over_ranks_two_gloo_processes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    # slowest rank's time (15 ms) and all ranks' tokens (7 + 14)
    assert got == [(0, 15.0, 21), (1, 15.0, 21)]


def test_reduce_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.5, 9, 1) == (3.5, 9)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_f32_e2e", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
