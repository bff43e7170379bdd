"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the path has no exchange
step, so ranks are independent replicas; the job time is the slowest rank's and the work
is the sum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from mixed_precision_kv_balancer_gb300 import inputs
    wl = inputs.WORKLOADS["tiny"].scaled(B=1, T=16)
    seeded = bench.rank_seed(wl, rank)
    x = inputs.make_prefill(seeded, 0, "cpu")["q"]
    ms = bench.reduce_over_ranks(10.0 + rank, world)
    out[rank] = (ms, float(x.float().sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_are_independent_replicas_timed_by_the_slowest():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 11.0          # max over ranks
    assert out[0][1] != out[1][1]                  # each rank draws its own sequences
    import bench
    assert bench.reduce_over_ranks(3.5, 1) == 3.5
