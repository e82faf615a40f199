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


def test_kernel_sources_cover_each_candidate():
    """bench.py trusts a candidate's committed ncu counters only while the
    hash of that candidate's kernel sources is unchanged, so each candidate
    must map to the file that defines it: where a candidate's name is a
    string literal in kernel files (its configuration table, or a table
    that refers to it), at least one of them is among the files hashed."""
    import re

    import matmul_selection_gb300 as mm

    kdir = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "matmul_selection_gb300", "csrc", "kernels")
    texts = {f: open(os.path.join(kdir, f)).read() for f in os.listdir(kdir) if f.endswith(".cu")}
    for name in mm.candidate_names():
        hashed = {os.path.basename(p) for p in bench.kernel_sources(name)}
        assert hashed and all(os.path.exists(os.path.join(kdir, f)) for f in hashed), name
        defining = {f for f, t in texts.items() if re.search(r'"%s"' % re.escape(name), t)}
        assert not defining or defining & hashed, (name, sorted(defining), sorted(hashed))
