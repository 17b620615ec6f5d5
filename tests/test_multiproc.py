"""The N > 1 bench path on CPU: replicas of the layer on 2 gloo ranks.  Every rank
reports its own time; the job's time is the slowest rank's and its throughput
counts every rank's tokens (weak scaling, no data exchange between replicas)."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 100.0 + 25.0 * rank            # rank 1 is the slower replica
        slowest = bench.max_over_ranks(my_ms)
        value = bench.replica_throughput(world, 8192, 10, slowest)
        q.put((rank, slowest, value, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, 29517
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, env in out:
        assert slowest == 125.0
        assert value == pytest.approx(2 * 8192 * 10 / 0.125)
        assert env == (2, rank, 0)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.replica_throughput(1, 100, 10, 1000.0) == pytest.approx(1000.0)
