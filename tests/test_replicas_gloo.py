"""Multi-GPU is replicas only (the tick has no cross-session exchange): each rank runs
its own sessions and bench.py aggregates whole-job throughput as all ranks'
session-frames over the slowest rank's time.  Checked with two gloo ranks on CPU."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [120.0, 150.0][rank]          # each rank's timed region
    frames = [64 * 10, 64 * 10][rank]  # each rank's session-frames
    tmax = bench.max_over_ranks(world, ms)
    total = bench.sum_over_ranks(world, frames)
    bench.barrier(world)
    q.put((rank, tmax, total, total / (tmax / 1000.0)))
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, tmax, total, value in res:
        assert tmax == 150.0 and total == 1280
        assert abs(value - 1280 / 0.150) < 1e-6
