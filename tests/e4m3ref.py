"""Host reference of the e4m3 output-layer quantization (test infrastructure).

The RNNT_BF16_E4M3 dtype computes the output layer with W^O_q, W^O quantized
per block of 256 rows to e4m3 with a power-of-two scale (include/rnnt.h,
rnnt_dims.dtype).  The oracle is fed W^O_q, so the tests need it on the host,
computed independently of the CUDA library: the block scale from the block's
largest magnitude, and the rounding by PyTorch's own float8_e4m3fn conversion.
"""
from __future__ import annotations

import math

import torch

E4M3_MAX = 448.0
BLOCK = 256
Z_SCALE = 256.0


def block_scale(amax: float) -> float:
    """The smallest power of two S with amax / S <= 448 (1 for amax = 0)."""
    if amax == 0.0:
        return 1.0
    k = math.ceil(math.log2(amax / E4M3_MAX))
    # guard the floating-point log at exact powers of two
    while amax / 2.0 ** k > E4M3_MAX:
        k += 1
    while amax / 2.0 ** (k - 1) <= E4M3_MAX:
        k -= 1
    return 2.0 ** k


def quantize_wo(WO: torch.Tensor):
    """(q bytes [V,H] uint8, W^O_q [V,H] float64, scales [ceil(V/256)] float64)."""
    W = WO.double()
    V = W.shape[0]
    q = torch.empty(W.shape, dtype=torch.uint8)
    Wq = torch.empty_like(W)
    scales = []
    for b0 in range(0, V, BLOCK):
        blk = W[b0:b0 + BLOCK]
        S = block_scale(float(blk.abs().max()))
        scales.append(S)
        f8 = (blk / S).float().to(torch.float8_e4m3fn)   # exact division by 2^k
        q[b0:b0 + BLOCK] = f8.view(torch.uint8)
        Wq[b0:b0 + BLOCK] = f8.double() * S
    return q, Wq, torch.tensor(scales, dtype=torch.float64)


def with_quantized_wo(inp):
    """A copy of synthetic inputs whose W^O is W^O_q (bf16; exact)."""
    import copy
    out = copy.copy(inp)
    _, Wq, _ = quantize_wo(inp.WO)
    out.WO = Wq.to(torch.bfloat16)
    assert torch.equal(out.WO.double(), Wq), "W^O_q is not exact in bf16"
    return out
