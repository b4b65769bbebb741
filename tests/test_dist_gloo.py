"""Multi-rank host logic of bench.py on CPU: two gloo ranks, no GPU.

The path shards by batch with no data exchange (every rank runs its own
replica), so the only cross-rank step is the timing reduction: the slowest
rank's time sets the whole-job throughput.
"""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_time = [2.0, 3.5][rank]
        slowest = bench.reduce_max(local_time, world, torch.device("cpu"))
        value = bench.aggregate_value(16384, 10, world, slowest)
        out[rank] = (slowest, value, bench.rank_seed(7, rank))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == 3.5
    assert out[0][1] == out[1][1] == pytest.approx(2 * 16384 * 10 / 3.5)
    assert out[0][2] != out[1][2]          # each replica draws its own batch


def test_single_rank_needs_no_group():
    assert bench.reduce_max(1.25, 1, torch.device("cpu")) == 1.25
    assert bench.aggregate_value(100, 4, 1, 2.0) == 200.0
