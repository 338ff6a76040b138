"""Multi-process host logic of bench.py on CPU: two gloo ranks, each timing
its own replica, agree on the slowest rank's time and on the whole-job
throughput (no GPU)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 100.0 + 25.0 * rank          # rank 1 is the slowest
        slowest = bench.max_over_ranks(mine)
        dist.barrier()
        results[rank] = (slowest, bench.job_throughput(world, 50, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_use_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == results[1]
    slowest, value = results[0]
    assert slowest == 125.0
    assert value == pytest.approx(2 * 50 / 0.125)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(1, 10, 20.0) == pytest.approx(500.0)
