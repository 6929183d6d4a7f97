"""The multi-GPU path is replicas only: N independent layers, one per rank, no data-path collective.

What bench.py does across ranks is host logic -- the slowest rank's time is the job's time, and the
job's rate counts every rank's units -- so it runs here on CPU as a 2-rank gloo group.
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


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 * (rank + 1)                 # rank 1 is the slower replica
        job_ms = bench.max_over_ranks(ms, torch.device("cpu"))
        rate = bench.whole_job_rate(1024, world, job_ms / 1)
        dist.barrier()
        out[rank] = (job_ms, rate)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_time_and_sum_the_work():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    job_ms, rate = out[0]
    assert job_ms == 20.0
    assert rate == pytest.approx(2 * 1024 / 0.020)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.whole_job_rate(100, 1, 10.0) == pytest.approx(10000.0)
