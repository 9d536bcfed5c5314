"""The benchmark's multi-rank bookkeeping on CPU (gloo, two ranks): the job's
time is the slowest rank's, every rank sees it, and throughput counts every
replica's weights.  The products themselves run as independent replicas (no
data-path collective), so this is all the N > 1 path adds."""
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
        ms = [1.25, 2.5][rank]  # rank 1 is the slow replica
        out[rank] = bench.max_over_ranks(torch, dist, ms, "cpu")
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_process_and_job_throughput():
    assert bench.max_over_ranks(torch, None, 3.0, "cpu") == 3.0
    # two replicas of 2.49 GB per step in 1.0 ms: 4980 GB/s for the job
    assert bench.job_gbs(2.49e9, 2, 1.0) == pytest.approx(4980.0)
    assert bench.job_gbs(2.49e9, 1, 1.0) == pytest.approx(2490.0)
