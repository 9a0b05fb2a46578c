"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks.

Each rank runs its own replica (no data-path collective); the only exchange is
the timing reduction, which must give every rank the slowest rank's time, and
the job throughput must count every rank's work."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        mine = 1.0 + 0.5 * rank                     # rank 1 is the slow one
        worst = bench.max_over_ranks(mine, ws)
        dist.barrier()
        out[rank] = worst
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 1.5, 1: 1.5}


def test_job_throughput_counts_every_replica():
    import bench
    one = bench.job_throughput(2e12, 1, 1.0)
    assert one == pytest.approx(2000.0)
    assert bench.job_throughput(2e12, 4, 1.0) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.25, 1) == 3.25
