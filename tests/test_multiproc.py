"""Host logic of multi-GPU runs on CPU (gloo, world size 2).  The layer shards trivially:
each rank runs independent replicas of the workload, no collective touches the data path;
ranks only meet at the timing barriers and the max-over-ranks reduction, and the whole-job
throughput counts every rank's tokens over the slowest rank's time."""
import os
import socket

import pytest
import torch
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
    w, r, l = bench.dist_env()
    assert (w, r, l) == (world, rank, rank)
    bench.barrier(world)
    my_seconds = 0.5 + rank  # rank 1 is the slowest
    slowest = bench.max_over_ranks(my_seconds, world, "cpu")
    value = bench.aggregate(256, 10, world, slowest)
    out[rank] = (slowest, value)
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_rank_timing_reduction_and_aggregate():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this (threaded) process
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, value = res[rank]
        assert slowest == pytest.approx(1.5)
        assert value == pytest.approx(256 * 10 * world / 1.5)


def test_single_rank_defaults():
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0
    assert bench.aggregate(100, 4, 1, 2.0) == 200.0
