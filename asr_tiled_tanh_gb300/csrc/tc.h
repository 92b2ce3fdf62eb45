// tc.h -- bf16 tensor-core (tcgen05 / TMEM / TMA) path of librnnt_gb300 (internal).
#pragma once
#include <functional>
#include "common.cuh"

namespace rnnt {

// RNNT_OK or RNNT_ERR_UNSUPPORTED_SHAPE for shapes the tensor-core kernels cannot take.
rnnt_status tc_check_shape(const Plan& p);
// out[M,H] = X[M,K] W[H,K]^T (+ bias[H]), bf16 operands, fp32 result.
cudaError_t tc_projection(const Plan& p, const void* X, const void* W, const void* bias, int M,
                          int K, float* out, cudaStream_t s);
// The e4m3 score GEMMs' operands (dtype RNNT_BF16_E4M3): z8, the chunk's
// e4m3(2^8 z) rows [rows][H]; wo8, W^O quantized per 256-row block [V][H];
// wodq, the dequantized W^O_q [V][H] bf16 (the backward's dz operand);
// nscale, the per-block factor of the accumulators.  NULL: bf16 scores.
struct TcF8 {
  unsigned char* z8;
  const void* wo8;
  const void* wodq;
  const float* nscale;
};
// wo8, wodq and nscale of TcF8 from W^O (bf16 [V][H]).
cudaError_t tc_quantize_wo(const Plan& p, const void* WO, void* wo8, void* wodq, float* nscale,
                           cudaStream_t s);
// Forward over every tile: lnPD, lpb, lpl into saved.  Z is the z buffer (the
// tile workspace, or the kept z in untiled mode); Hkeep, when given, receives
// the scores (untiled mode).
rnnt_status tc_forward_tiles(const Plan& p, const SavedView& sv, const rnnt_params* pr,
                             const int32_t* labels, const int32_t* T_len, const int32_t* U_len,
                             const float* pA, const float* pL, void* Z, void* Hkeep,
                             const TcF8* f8, cudaStream_t s);
// Backward over every tile: dA, dLr (accumulated), dW^O, db^O.  post: the
// per-row posterior records of one chunk (chunk_rows float4, tiled mode).
// Launches a caller has the backward make: `pre` on a side stream while the
// first chunk's z is rebuilt (they must be done before the chunk's dh
// kernel), `after` once the last chunk's dz is done (it may read dA, dLr),
// beside that chunk's dW^O.  z_resident: Z already holds the z tiles of a
// single-chunk plan (built by the forward of the same call), which are then
// not rebuilt.
using PreLaunch = std::function<rnnt_status(cudaStream_t)>;
rnnt_status tc_backward_tiles(const Plan& p, const SavedView& sv, const rnnt_params* pr,
                              const int32_t* labels, const int32_t* T_len, const int32_t* U_len,
                              const float* grad_loss, const float* pA, const float* pL, void* Z,
                              void* Hs, bool untiled, bool z_resident, float* dA, float* dLr,
                              float* dWO,
                              float* dbO, float4* post, const TcF8* f8, const PreLaunch* pre,
                              const PreLaunch* after, cudaStream_t s);
// How the encoder-side gradients leave (rnnt_bwd_ex): bf16: dhA, dhL (and
// dA, dL) are bf16, else fp32; dA, dL: the projections' gradients, or NULL.
struct EncOut {
  bool bf16;
  void* dA;
  void* dL;
};
// dh^A, dW^A, dh^L, dW^L, db^Z from dA and dLr.
rnnt_status tc_encoder_grads(const Plan& p, char* ws, const void* hA, const void* hL,
                             const rnnt_params* pr, const int32_t* Teff, const int32_t* Ueff,
                             float* dA, float* dLr, void* dhA, void* dhL, float* dWA,
                             float* dWL, float* dbZ, const EncOut& out, cudaStream_t s);

}  // namespace rnnt
