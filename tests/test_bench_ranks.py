"""The replicas-only multi-rank path of bench.py on CPU (gloo, two ranks):
the slowest rank's time is every rank's, and the whole-job rate counts the
work of all replicas."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as tmp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank  # rank 1 is the slower replica
        t = bench.max_over_ranks(mine, world, "cpu")
        out[rank] = (t, bench.aggregate_rate(100.0, world, t))
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    out = tmp.Manager().dict()
    tmp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == (15.0, 100.0 * 2 / 15.0)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.aggregate_rate(10.0, 1, 2.0) == 5.0
