"""The N > 1 path of bench.py on CPU: independent replicas, one process per rank, with
the job time taken as the maximum over ranks (gloo, world size 2, 127.0.0.1)."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, rank, world)
        ms_local = 100.0 + 50.0 * rank          # rank 1 is the slow one
        ms, per_s = bench.aggregate_over_ranks(ms_local, 1e12, 10, world,
                                               bench.torch_all_reduce_max("cpu"))
        out[rank] = (ms, per_s)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world = 2
    out = mp.get_context("spawn").Manager().dict()   # no fork of this multi-threaded process
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        ms, per_s = out[rank]
        assert ms == 150.0                       # every rank sees the slowest rank's time
        assert per_s == pytest.approx(1e12 * 10 * world / 0.150)


def test_single_process_needs_no_collective():
    ms, per_s = bench.aggregate_over_ranks(200.0, 5.0, 4, 1, None)
    assert ms == 200.0 and per_s == pytest.approx(5.0 * 4 / 0.2)
