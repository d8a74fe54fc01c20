"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): the
job's time is the slowest rank's and its throughput counts every rank's
tokens (weak scaling, one replica per rank, no data-path collective)."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = [100.0, 250.0][rank]  # rank 1 is the slow one
        value, ms = bench.job_throughput(ms_local, tokens_per_rank=1000, steps=10, dist=dist)
        out[rank] = (value, ms)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_throughput_single_rank():
    value, ms = bench.job_throughput(50.0, tokens_per_rank=2000, steps=5)
    assert ms == 50.0
    assert value == pytest.approx(2000 / (50.0 / 5 / 1e3))


def test_job_throughput_two_gloo_ranks_take_the_slowest_rank():
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:  # no fork of a multi-threaded parent
        out = mgr.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        value, ms = res[rank]
        assert ms == 250.0
        assert value == pytest.approx(2 * 1000 / (250.0 / 10 / 1e3))
