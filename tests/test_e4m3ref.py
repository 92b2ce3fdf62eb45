"""The host e4m3 quantization reference against facts of the format (CPU).

e4m3 (the float8 "fn" variant): 1 sign, 4 exponent (bias 7) and 3 mantissa
bits, no infinities, largest finite 448, smallest normal 2^-6, smallest
subnormal 2^-9, round to nearest even.
"""
import math

import pytest
import torch

from tests import e4m3ref


def _e4m3(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).float().tolist()


def test_representable_points_and_ties():
    assert _e4m3([448.0, 1.0, 1.125, 2.0 ** -6, 2.0 ** -9]) == [448.0, 1.0, 1.125, 2.0 ** -6,
                                                                2.0 ** -9]
    # ties go to the even mantissa: 1.0625 between 1.0 (000) and 1.125 (001)
    # -> 1.0; 1.1875 between 1.125 (001) and 1.25 (010) -> 1.25
    assert _e4m3([1.0625, 1.1875, -1.0625]) == [1.0, 1.25, -1.0]
    # spacing 2^(e-3) in the binade [2^e, 2^(e+1)): 240 -> 240, 250 -> 256
    assert _e4m3([240.0, 250.0, 0.3]) == [240.0, 256.0, 0.3125]


@pytest.mark.parametrize("amax,S", [(448.0, 1.0), (449.0, 2.0), (0.224, 2.0 ** -10),
                                    (0.0, 1.0), (896.0, 2.0), (896.5, 4.0), (1.0, 2.0 ** -8)])
def test_block_scale_is_the_smallest_fitting_power_of_two(amax, S):
    assert e4m3ref.block_scale(amax) == S
    if amax > 0:
        assert amax / S <= 448.0 < amax / (S / 2)


def test_quantized_output_layer_properties():
    g = torch.Generator().manual_seed(5)
    V, H = 600, 48   # three blocks, the last one ragged
    WO = (torch.randn(V, H, generator=g) / math.sqrt(H)).to(torch.bfloat16)
    WO[256:512] *= 40.0          # blocks with different ranges
    q, Wq, scales = e4m3ref.quantize_wo(WO)
    assert scales.numel() == 3
    for b, S in enumerate(scales.tolist()):
        assert S == 2.0 ** round(math.log2(S))                 # powers of two
        blk = WO[b * 256:(b + 1) * 256].double()
        assert blk.abs().max() / S <= 448.0
        qs = Wq[b * 256:(b + 1) * 256] / S
        assert qs.abs().max() <= 448.0
        # normal values keep 3 mantissa bits: relative error <= 2^-4
        big = blk.abs() >= 2.0 ** -6 * S
        rel = ((Wq[b * 256:(b + 1) * 256] - blk).abs() / blk.abs())[big]
        assert rel.max() <= 2.0 ** -4 + 1e-12
    # W^O_q is exact in bf16 (4 significant bits times a power of two)
    assert torch.equal(Wq.to(torch.bfloat16).double(), Wq)
    # the bytes decode to W^O_q / S
    dec = q.view(torch.float8_e4m3fn).double()
    for b, S in enumerate(scales.tolist()):
        assert torch.equal(dec[b * 256:(b + 1) * 256] * S, Wq[b * 256:(b + 1) * 256])
