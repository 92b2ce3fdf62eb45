"""Data-parallel sharding of a transducer batch over ranks (one process per GPU).

The samples of a batch are independent lattices: the loss is a sum over
samples (sample-wise paper §2, Eq. 9) and the parameter gradients are sums of
per-sample contributions (the sample-wise paper §4: accumulating sample by
sample equals the batched computation).  So a batch splits across ranks by
samples with no exchange during the forward or backward pass; the one
collective is a sum of the parameter gradients (dW^A, dW^L, db^Z, dW^O, db^O)
after each rank's backward.  The per-sample outputs (loss, dh^A, dh^L) stay on
the rank that owns the sample.  The Flash RNN-T blog's measurements ("What
changed in practice") ran data-parallel on 8 GPUs in this way.

This module holds the host side of that arrangement: which samples a rank
owns, and one flat buffer for the parameter gradients so that the sum is a
single all-reduce.  The reduction itself is torch.distributed's (NCCL between
GPUs, gloo on CPU ranks); the library's kernels fill the buffer.
"""
from __future__ import annotations

import torch

# Parameter gradients, in their order inside the flat buffer.
PARAM_GRADS = ("dWA", "dWL", "dbZ", "dWO", "dbO")
# Per-sample gradients (not reduced: each rank keeps its samples').
SAMPLE_GRADS = ("dhA", "dhL")


def shard_range(B: int, rank: int, world: int) -> tuple[int, int]:
    """Samples [lo, hi) of a batch of B owned by `rank` of `world`: contiguous
    ranges whose sizes differ by at most one (the first B % world ranks take
    one more)."""
    if world < 1 or not 0 <= rank < world or B < 0:
        raise ValueError(f"shard_range(B={B}, rank={rank}, world={world})")
    base, extra = divmod(B, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def param_grad_shapes(H: int, HA: int, HL: int, V: int) -> dict:
    return {"dWA": (H, HA), "dWL": (H, HL), "dbZ": (H,), "dWO": (V, H), "dbO": (V,)}


def alloc_grads(B: int, T: int, U1: int, HA: int, HL: int, H: int, V: int,
                device="cuda") -> tuple[torch.Tensor, dict]:
    """Gradient buffers for one rank: the parameter gradients as views into
    one flat fp32 buffer (returned first, for the all-reduce), the per-sample
    ones as their own tensors.  The views keep the 16-byte alignment the
    library's vector reductions use (every offset is a multiple of 4 floats)."""
    shapes = param_grad_shapes(H, HA, HL, V)
    sizes = {k: int(torch.Size(shapes[k]).numel()) for k in PARAM_GRADS}
    offs, o = {}, 0
    for k in PARAM_GRADS:
        offs[k] = o
        o += (sizes[k] + 3) // 4 * 4
    flat = torch.zeros(o, dtype=torch.float32, device=device)
    grads = {k: flat[offs[k]:offs[k] + sizes[k]].view(shapes[k]) for k in PARAM_GRADS}
    f = dict(dtype=torch.float32, device=device)
    grads["dhA"] = torch.empty(B, T, HA, **f)
    grads["dhL"] = torch.empty(B, U1, HL, **f)
    return flat, grads


def allreduce_param_grads(flat: torch.Tensor, dist=None, group=None) -> None:
    """Sum the flat parameter-gradient buffer over the ranks of `group` (in
    place, on the current stream).  A no-op without a process group."""
    if dist is None or not dist.is_initialized() or dist.get_world_size(group) == 1:
        return
    dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
