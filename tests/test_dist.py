"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the timed region is the
slowest rank's, and the whole-job throughput counts every rank's units. The benchmark runs
independent replicas per GPU, so there is no data-path collective to test."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    bench.init_dist(world, "gloo")
    t = bench.max_over_ranks(1.5 + rank, world)          # rank 1 is the slowest
    v = bench.aggregate_throughput(1000.0, t, world)
    bench.barrier(world)
    out[rank] = (t, v)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_and_aggregate():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        t, v = out[rank]
        assert t == 2.5                                    # max over ranks
        assert v == pytest.approx(1000.0 * 2 / 2.5)        # all ranks' units / slowest time


def test_single_rank_helpers_are_identity():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.aggregate_throughput(10.0, 2.0, 1) == 5.0
