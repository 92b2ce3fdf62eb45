/*
 * rnnt_testing.h -- test hook of librnnt_gb300 (not part of the method).
 *
 * Exposes the library's bf16 tcgen05 GEMM kernel on its own so that its
 * operand layouts can be checked against a host matrix product.
 */
#ifndef RNNT_GB300_TESTING_H
#define RNNT_GB300_TESTING_H

#include "rnnt.h"

#ifdef __cplusplus
extern "C" {
#endif

/* C[M,N] (fp32, row-major, leading dimension N) = op(A) op(B), bf16 device
 * operands: A is [M,K] row-major (a_mn = 0) or [K,M] row-major (a_mn = 1);
 * B is [N,K] row-major (b_mn = 0, i.e. C = A B^T) or [K,N] row-major
 * (b_mn = 1).  accumulate = 0: C is overwritten (k_splits ignored);
 * accumulate = 1: the product is added to C with fp32 atomics, K split into
 * k_splits ranges.  bn: 128 or 256 (the kernel's N tile).  The contiguous
 * extent of each operand must be a multiple of 8 elements and the pointers
 * 16-byte aligned.  Asynchronous on `stream` (a cudaStream_t). */
rnnt_status rnnt_testing_gemm_bf16(int M, int N, int K, const void* A, int a_mn, const void* B,
                                   int b_mn, float* C, int accumulate, int k_splits, int bn,
                                   void* stream);

/* Failure-detection hook: the same GEMM (A [M,K], B [N,K], both K-major,
 * C = A B^T) with the first pipeline stage never filled, so the kernel's
 * bounded mbarrier waits run out after `wait_ns` nanoseconds each.  The
 * kernel then sets bit RNNT_ERR_TIMEOUT in the device int32 `*status`, stops
 * issuing work, waits (bounded) for the loads it did issue, frees its TMEM
 * and returns; nothing traps and the CUDA context stays usable.  C is left
 * undefined.  Asynchronous on `stream`. */
rnnt_status rnnt_testing_gemm_timeout(int M, int N, int K, const void* A, const void* B,
                                      float* C, int32_t* status, unsigned long long wait_ns,
                                      void* stream);

/* The W^O quantization of the RNNT_BF16_E4M3 dtype on its own: WO bf16
 * [V,H] (device) -> Q e4m3 bytes [V,H], Wdq = the dequantized W^O_q bf16
 * [V,H], nscale fp32 [ceil(V/256)] = S / 2^8 per block of 256 rows (S: the
 * block's power-of-two scale, see rnnt_dims.dtype).  H must be even.
 * Asynchronous on `stream`. */
rnnt_status rnnt_testing_quantize_wo(int V, int H, const void* WO, void* Q, void* Wdq,
                                     float* nscale, void* stream);

#ifdef __cplusplus
}
#endif
#endif
