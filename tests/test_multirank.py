"""The bench's multi-rank bookkeeping on CPU ranks (gloo, world size 2): each
rank times its own replica of the layer, the job time is the slowest rank's,
and the job throughput counts every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, ms_of_rank, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(ms_of_rank[rank], world, torch.device("cpu"))
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_throughput_gloo():
    world = 2
    ms = [12.5, 17.25]
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), ms, out), nprocs=world, join=True,
                       start_method="spawn")
    assert [out[r] for r in range(world)] == [max(ms)] * world
    # 2 replicas of 1e12 FLOPs in the slowest rank's 17.25 ms
    assert bench.job_throughput(1e12, world, max(ms)) == pytest.approx(2e12 / 17.25e-3 / 1e12)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
