"""Multi-rank bench logic on the CPU (gloo, world size 2): with N replicas the step
time reported is the max over ranks, so the slowest replica sets the number."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (world, rank, rank)
        bench.barrier(world)
        out[rank] = bench.max_over_ranks(1.5 + 2.0 * rank, world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    world = 2
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
        assert dict(out) == {0: 3.5, 1: 3.5}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(2.25, 1) == 2.25
    bench.barrier(1)
