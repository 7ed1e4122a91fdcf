"""The benchmark's multi-rank bookkeeping (max time over ranks, summed
launches, whole-job throughput) on two gloo ranks on the CPU, and the
reference arm's rank-0-only rule."""

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


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, n = bench.reduce_over_ranks(100.0 + 25.0 * rank, 500 + rank, "cpu")
        q.put((rank, ms, n, bench.job_tokens_per_s(world, 32768, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_time_and_sum_launches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, n, tps in got:
        assert ms == 125.0          # the slower rank's time
        assert n == 1001            # launches of both ranks
        assert abs(tps - 2 * 32768 / 0.125) < 1e-6


def test_reference_arm_prints_nothing_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
