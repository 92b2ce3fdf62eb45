"""The multi-rank bookkeeping of bench.py on CPU ranks (gloo, world size 2).

Each rank runs its own batch; the job time is the slowest rank's and the job
value counts every rank's cells.
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank
    got = bench.reduce_max(ms, dist, torch.device("cpu"))
    out[rank] = (got, bench.job_value(1000, world, got))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == (15.0, 2000 / 0.015)


def test_single_rank_needs_no_process_group():
    assert bench.reduce_max(3.5, None, None) == 3.5
    assert bench.job_value(500, 1, 2.0) == 250000.0
