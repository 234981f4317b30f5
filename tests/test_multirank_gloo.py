"""The multi-rank path of bench.py on CPU: two gloo ranks reduce their timings.

The decode path shards without any exchange (independent requests and KV heads),
so N ranks run N independent replicas; the job's time is the slowest rank's and
its throughput is every rank's bytes over that time.  This checks the reduction
with two processes on the gloo backend, and that the reference arm only prints
on rank 0.
"""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, units = bench.reduce_over_ranks(10.0 + 5.0 * rank, 1000.0 * (rank + 1), world)
        q.put((rank, ms, units))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_sum_the_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    assert got == [(0, 15.0, 3000.0), (1, 15.0, 3000.0)]


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(7.5, 42.0, 1) == (7.5, 42.0)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0 and res.stdout.strip() == ""
