"""The bench's multi-rank path on CPU (gloo, world size 2): every rank runs its
own copy of the workload (the units are independent, no data-path collective),
the timing is the maximum over ranks, and the reported value is the whole-job
throughput."""
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
        mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(mine, dist)
        out[rank] = slowest
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork after torch has started threads
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == 15.0 and out[1] == 15.0


def test_job_throughput_and_single_rank():
    assert bench.max_over_ranks(3.5, None) == 3.5
    # 2 ranks x 65536 tokens x 10 steps in 20 ms (slowest rank)
    assert bench.job_tokens_per_s(2, 65536, 10, 20.0) == pytest.approx(2 * 65536 * 10 / 0.02)
