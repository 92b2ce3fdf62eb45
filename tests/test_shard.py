"""Data-parallel sharding on CPU ranks (gloo, world size 2).

A batch split by samples over two ranks, each rank's gradients computed on its
samples alone and the parameter gradients summed by the one all-reduce of
asr_tiled_tanh_gb300.shard, gives the gradients of the whole batch: the loss is
a sum over samples (sample-wise paper §2, Eq. 9) and the method accumulates
parameter gradients sample by sample (§4).  The per-rank arithmetic here is the
oracle's (no GPU); the host logic under test is the sharding and the reduction.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from asr_tiled_tanh_gb300 import shard, synthetic
from tests.helpers import run_oracle


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    # B = 5 over two ranks: shards of 3 and 2 samples, mixed lengths, biases
    return synthetic.custom(B=5, T=7, U=3, HA=6, HL=5, H=8, V=7, dtype="f32", seed=11,
                            bias_std=0.2)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    torch.set_num_threads(1)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = _inputs()
    wl = inp.wl
    lo, hi = shard.shard_range(wl.B, rank, world)
    mine = inp.subset(list(range(lo, hi)))
    o = run_oracle(mine, nthreads=1)
    flat, grads = shard.alloc_grads(hi - lo, wl.T, wl.U1, wl.HA, wl.HL, wl.H, wl.V, device="cpu")
    for k in shard.PARAM_GRADS:
        grads[k].copy_(torch.from_numpy(o.grads[k]))
    shard.allreduce_param_grads(flat, dist)
    out[rank] = dict(lo=lo, hi=hi, loss=o.loss.copy(),
                     dhA=o.grads["dhA"].copy(), dhL=o.grads["dhL"].copy(),
                     **{k: grads[k].numpy().copy() for k in shard.PARAM_GRADS})
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_gradients_all_reduced_equal_the_whole_batch():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = {r: dict(v) for r, v in out.items()}
    full = run_oracle(_inputs())
    assert (res[0]["lo"], res[0]["hi"], res[1]["lo"], res[1]["hi"]) == (0, 3, 3, 5)
    # per-sample outputs stay with their rank and concatenate to the batch's
    np.testing.assert_allclose(np.concatenate([res[0]["loss"], res[1]["loss"]]), full.loss,
                               rtol=1e-12)
    for k in shard.SAMPLE_GRADS:
        np.testing.assert_allclose(np.concatenate([res[0][k], res[1][k]]), full.grads[k],
                                   rtol=1e-12, atol=1e-15)
    # every rank holds the summed parameter gradients (fp32 buffer)
    for rank in (0, 1):
        for k in shard.PARAM_GRADS:
            ref = full.grads[k]
            err = np.linalg.norm(res[rank][k] - ref) / np.linalg.norm(ref)
            assert err < 1e-6, (rank, k, err)
    for k in shard.PARAM_GRADS:
        assert np.array_equal(res[0][k], res[1][k])


@pytest.mark.parametrize("B", [0, 1, 2, 5, 8, 1023, 1024])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shard_ranges_cover_the_batch_once(B, world):
    ranges = [shard.shard_range(B, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == B
    for (lo0, hi0), (lo1, hi1) in zip(ranges, ranges[1:]):
        assert hi0 == lo1
    sizes = [hi - lo for lo, hi in ranges]
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0


def test_flat_gradient_views_are_aligned_and_disjoint():
    flat, g = shard.alloc_grads(2, 5, 4, 12, 10, 9, 13, device="cpu")
    spans = []
    for k in shard.PARAM_GRADS:
        off = (g[k].data_ptr() - flat.data_ptr()) // 4
        assert off % 4 == 0, k                       # 16-byte aligned within the buffer
        spans.append((off, off + g[k].numel()))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    assert spans[-1][1] <= flat.numel()
    assert g["dWO"].shape == (13, 9) and g["dbO"].shape == (13,) and g["dhA"].shape == (2, 5, 12)


def test_single_rank_reduction_is_a_no_op():
    flat, _ = shard.alloc_grads(1, 2, 2, 4, 4, 4, 4, device="cpu")
    flat.fill_(1.5)
    shard.allreduce_param_grads(flat, None)
    assert torch.all(flat == 1.5)
