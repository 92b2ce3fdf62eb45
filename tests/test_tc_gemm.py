"""The tcgen05 GEMM kernel on its own, against a host fp64 product (GPU).

Every operand layout the library uses (A and B each K-major or MN-major),
both N tiles, overwrite and split-K atomic accumulation, with M, N and K that
are not multiples of the 128 x BN x 64 tile.
"""
import itertools

import pytest
import torch

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rn.load(build_if_missing=True)


def _case(M, N, K, a_mn, b_mn, seed):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)   # C = A B^T
    ref = A.double() @ B.double().T
    A_dev = (A.T.contiguous() if a_mn else A).cuda()
    B_dev = (B.T.contiguous() if b_mn else B).cuda()
    return A_dev, B_dev, ref


@pytest.mark.parametrize("a_mn,b_mn,bn", list(itertools.product([0, 1], [0, 1], [128, 256])))
def test_gemm_layouts_store(a_mn, b_mn, bn):
    M, N, K = 328, 200, 200
    A, B, ref = _case(M, N, K, a_mn, b_mn, 1 + 4 * a_mn + 2 * b_mn)
    C = torch.full((M, N), float("nan"), device="cuda")
    binding.rnnt_testing_gemm_bf16(A, a_mn, B, b_mn, C, M, N, K, accumulate=0, bn=bn)
    torch.cuda.synchronize()
    err = (C.double().cpu() - ref).abs().max().item()
    assert err < 1e-3 * K ** 0.5, err


@pytest.mark.parametrize("a_mn,b_mn", list(itertools.product([0, 1], [0, 1])))
def test_gemm_layouts_split_k_atomic(a_mn, b_mn):
    M, N, K = 256, 136, 1000
    A, B, ref = _case(M, N, K, a_mn, b_mn, 11 + a_mn + 2 * b_mn)
    C = torch.ones((M, N), device="cuda")
    binding.rnnt_testing_gemm_bf16(A, a_mn, B, b_mn, C, M, N, K, accumulate=1, k_splits=5,
                                   bn=128)
    torch.cuda.synchronize()
    err = (C.double().cpu() - 1.0 - ref).abs().max().item()
    assert err < 1e-3 * K ** 0.5, err


def test_gemm_many_tiles_persistent():
    # more output tiles than SMs: every CTA walks several units
    M, N, K = 128 * 40, 512, 320
    A, B, ref = _case(M, N, K, 0, 0, 99)
    C = torch.empty((M, N), device="cuda")
    binding.rnnt_testing_gemm_bf16(A, 0, B, 0, C, M, N, K, bn=256)
    torch.cuda.synchronize()
    err = (C.double().cpu() - ref).abs().max().item()
    assert err < 1e-3 * K ** 0.5, err
    # the same product again with 128-wide N tiles (twice the units per CTA):
    # each output element is one K-ordered fp32 accumulation either way
    C2 = torch.empty((M, N), device="cuda")
    binding.rnnt_testing_gemm_bf16(A, 0, B, 0, C2, M, N, K, bn=128)
    torch.cuda.synchronize()
    assert torch.equal(C, C2)
