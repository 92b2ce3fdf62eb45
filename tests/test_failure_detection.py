"""Failure detection on the GPU without a fault (GPU).

Every mbarrier wait in the tensor-core kernels is bounded.  A test hook runs
the GEMM kernel with one pipeline stage that is never filled, so the MMA
thread's wait runs out: the kernel must record RNNT_ERR_TIMEOUT in the status
word, wind down (bounded waits for its own loads, TMEM freed) and return, and
the CUDA context must still compute correctly afterwards.
"""
import time

import pytest
import torch

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rn.load(build_if_missing=True)


def test_bounded_wait_reports_timeout_and_context_survives():
    g = torch.Generator().manual_seed(3)
    M, N, K = 256, 256, 512
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    C = torch.zeros(M, N, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    binding.rnnt_testing_gemm_timeout(A, B, C, status, M, N, K, wait_ns=50_000_000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) & (1 << 6), "timeout bit not set"
    assert elapsed < 10.0
    # the context is intact: a normal GEMM still gives the right answer
    C2 = torch.empty(M, N, device="cuda")
    binding.rnnt_testing_gemm_bf16(A, 0, B, 0, C2, M, N, K, bn=128)
    torch.cuda.synchronize()
    ref = A.double().cpu() @ B.double().cpu().T
    assert (C2.double().cpu() - ref).abs().max().item() < 1e-3 * K ** 0.5
