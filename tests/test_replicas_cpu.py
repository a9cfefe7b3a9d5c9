"""Multi-rank host logic on CPU (gloo, world size 2): sharding, MAX-reduced
timing and the aggregate throughput the benchmark reports."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from forward_mode_flash_gb300 import replicas


def test_shard_covers_everything_once():
    for n in (0, 1, 7, 64, 65):
        for world in (1, 2, 3, 8):
            spans = [replicas.shard(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        replicas.shard(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_s = [1.5, 2.0][rank]  # rank 1 is the slowest
        m = replicas.max_over_ranks(local_s)
        v = replicas.aggregate_throughput(world, 10.0, 4, m)
        out[rank] = (m, v)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_reduction_and_throughput():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == (2.0, 2 * 10.0 * 4 / 2.0)


def test_single_process_is_identity():
    assert replicas.max_over_ranks(3.25) == 3.25
