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


def test_gpus_flag_starts_one_process_per_gpu(monkeypatch):
    # without a launcher, `bench.py --gpus N` starts N ranks itself through
    # torch.distributed.run on 127.0.0.1 with the same arguments
    calls = []
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: calls.append(cmd) or 0)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench.sys, "argv", ["bench.py", "--gpus", "4", "--steps", "7",
                                            "--warmup", "3"])
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert e.value.code == 0
    (cmd,) = calls
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert "--nproc-per-node=4" in cmd and cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-6:] == ["--gpus", "4", "--steps", "7", "--warmup", "3"]
    assert cmd[-7].endswith("bench.py")


def test_gpus_flag_under_a_launcher_runs_in_place(monkeypatch):
    # started by a launcher (WORLD_SIZE set), the rank runs its own work
    ran = []
    monkeypatch.setattr(bench, "run_gpu_bench", lambda args: ran.append(args.gpus))
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: pytest.fail("relaunched"))
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(bench.sys, "argv", ["bench.py", "--gpus", "2"])
    bench.main()
    assert ran == [2]
