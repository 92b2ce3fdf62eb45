"""Data-parallel sharding with the library's kernels (GPU, one device).

The ranks of a data-parallel job each run their own samples; the job's
parameter gradients are the sum of the ranks' (one all-reduce).  Here the
ranks' shares of a batch run one after the other on one GPU, each with its own
plan and buffers (no collective and no waiting between them), and the summed
parameter gradients, the per-sample losses and the per-sample gradients equal
the whole batch's: losses bit for bit (each lattice's forward is independent of
the batch), gradients to 1e-5 (atomic reductions in another order).
"""
import numpy as np
import pytest
import torch

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import shard, synthetic
from tests.helpers import rel_l2, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rn.load(build_if_missing=True)


def _run(inp):
    dev = to_device(inp)
    r = rn.Rnnt.for_inputs(inp, tile_cells=128 * 8)  # several chunks
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    args = (dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
    loss = r.fwd(*args)
    g = r.bwd(*args)
    torch.cuda.synchronize()
    assert r.status() == (0, 0)
    return loss.cpu().numpy(), {k: v.double().cpu().numpy() for k, v in g.items()}


@pytest.mark.parametrize("dtype,world", [("bf16", 2), ("bf16", 3), ("f32", 2)])
def test_shards_sum_to_the_whole_batch(dtype, world):
    H, V = (128, 256) if dtype == "bf16" else (64, 96)
    inp = synthetic.custom(B=7, T=50, U=12, HA=H, HL=H, H=H, V=V, dtype=dtype, seed=91,
                           bias_std=0.1)
    loss_all, g_all = _run(inp)
    loss = np.zeros_like(loss_all)
    summed = {k: np.zeros_like(g_all[k]) for k in shard.PARAM_GRADS}
    per_sample = {k: np.zeros_like(g_all[k]) for k in shard.SAMPLE_GRADS}
    for rank in range(world):
        lo, hi = shard.shard_range(inp.wl.B, rank, world)
        l_r, g_r = _run(inp.subset(range(lo, hi)))
        loss[lo:hi] = l_r
        for k in shard.PARAM_GRADS:
            summed[k] += g_r[k]
        for k in shard.SAMPLE_GRADS:
            per_sample[k][lo:hi] = g_r[k]
    np.testing.assert_array_equal(loss, loss_all)
    for k in shard.PARAM_GRADS:
        assert rel_l2(summed[k], g_all[k]) < 1e-5, k
    for k in shard.SAMPLE_GRADS:
        assert rel_l2(per_sample[k], g_all[k]) < 1e-5, k
