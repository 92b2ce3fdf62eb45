// kernels.h -- host launchers of the library's kernels (internal).
#pragma once
#include "common.cuh"

namespace rnnt {

// ---- lattice bookkeeping and the loss recursion (k_lattice.cu) -----------
// Multiprocessor count of the current device (cached per device; 152 when
// the query fails).
int num_sms();
cudaError_t launch_fill_f32(float* p, float v, size_t n, cudaStream_t s);
cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s);
// Zero up to 8 buffers (16-byte aligned pointers) in one launch; NULL entries are skipped.
struct ZeroList {
  void* p[8];
  size_t bytes[8];
  int n;
};
cudaError_t launch_zero_many(const ZeroList& z, cudaStream_t s);
// Validate lengths/labels, build the per-sample tile prefix sum, reset the
// status word, mark rejected samples (loss = lnP = NaN).
cudaError_t launch_index(const Shape& sh, const int32_t* labels, const int32_t* T_len,
                         const int32_t* U_len, SavedView sv, float* loss, cudaStream_t s);
// Table of every actual tile's coordinates (saved.tiles), from the prefix sum.
cudaError_t launch_tile_table(const Shape& sh, const int32_t* T_len, const int32_t* U_len,
                              SavedView sv, cudaStream_t s);
// alpha/beta wavefronts over every sample's lattice; writes lnP and loss.
// fast: approximate ex2/lg2 in logaddexp (bf16 path); else expf/log1pf.
cudaError_t launch_alpha_beta(const Shape& sh, const int32_t* T_len, const int32_t* U_len,
                              SavedView sv, float* loss, bool fast, cudaStream_t s);

// Effective lengths for masked contractions over encoder rows: T_len[b] and
// U_len[b]+1 for accepted samples, 0 for rejected ones.
cudaError_t launch_eff_lengths(const Shape& sh, SavedView sv, const int32_t* T_len,
                               const int32_t* U_len, int32_t* Teff, int32_t* Ueff,
                               cudaStream_t s);

// ---- fp32 FFMA path (k_simt.cu) -------------------------------------------
struct SimtGemm {
  int M, N, K;
  const void* A; long long sam, sak; int a_bf16;    // A(m,k) = A[m*sam + k*sak]
  const void* Bm; long long sbk, sbn; int b_bf16;   // B(k,n) = Bm[k*sbk + n*sbn]
  float* C; long long ldc;                          // C[m*ldc + n]
  float alpha; int accumulate;                      // C = alpha*AB (+ C if accumulate)
  const void* bias; int bias_bf16;                  // + bias[n] (may be NULL)
  // Optional K mask: k contributes iff (k % kperiod) < kmask_len[k / kperiod] + kmask_off.
  const int32_t* kmask_len; int kperiod; int kmask_off;
};
cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t s);

struct ChunkArgs {
  Shape sh;
  long long first_tile;   // global index of the chunk's first tile
  long long ntiles;       // tiles in the chunk buffer
  const int32_t* T_len;
  const int32_t* U_len;
  const int32_t* labels;
  SavedView sv;
};
// z rows of the chunk (fp32 or bf16): tanh(pA[b,t] + pL[b,u]); 0 on masked rows.
cudaError_t launch_build_z(const ChunkArgs& c, const float* pA, const float* pL, void* Z,
                           int z_bf16, cudaStream_t s);
// Row-wise log-sum-exp of fp32 scores; writes lnPD, lpb, lpl into saved.
cudaError_t launch_lse_rows(const ChunkArgs& c, const float* Hs, cudaStream_t s);
// dh over the fp32 scores in place (masked rows become 0).
cudaError_t launch_dh_rows(const ChunkArgs& c, float* Hs, const float* grad_loss,
                           cudaStream_t s);
// da = dz (1 - z^2) reduced into dA[b,t,:] and dLr[b,u,:] (fp32 atomics).
cudaError_t launch_da_reduce(const ChunkArgs& c, const float* dZ, const void* Z, int z_bf16,
                             float* dA, float* dLr, cudaStream_t s);
// out[n] (+)= sum_r X[r*ld + n] for r < R.
cudaError_t launch_colsum(const float* X, long long R, int N, long long ld, float* out,
                          cudaStream_t s);

// ---- chunk walk (api.cu) ----------------------------------------------------
// Number of chunks of tiles a pass walks: the upper bound when every possible
// tile fits one chunk (no synchronization); otherwise the actual tile count is
// read back from the device (one synchronization of st).
rnnt_status chunk_count(const Plan& p, const SavedView& sv, cudaStream_t st, long long* n);
// Arguments of chunk k (its first tile and the chunk buffer's tile count).
ChunkArgs chunk_args(const Plan& p, const SavedView& sv, long long k, const int32_t* labels,
                     const int32_t* T_len, const int32_t* U_len);

// ---- the forward pass behind rnnt_fwd (api.cu) ----------------------------
// side_streams: run the independent launches on side streams (false: every
// launch on `stream`, and no stream is ever created).
rnnt_status fwd_impl(const rnnt_dims* dims, const void* hA, const void* hL,
                     const rnnt_params* pr, const int32_t* labels, const int32_t* T_len,
                     const int32_t* U_len, float* loss, void* saved, void* ws, size_t ws_bytes,
                     rnnt_stream stream, bool side_streams);

// ---- the backward pass behind rnnt_bwd and rnnt_fwd_bwd (api.cu) -----------
// z_resident: the workspace still holds the z tiles the forward of the same
// call built, so that a single-chunk plan does not rebuild them.
// opts: the encoder-side hand-off of rnnt_bwd_ex (NULL: fp32 dhA, dhL).
rnnt_status bwd_impl(const rnnt_dims* dims, const void* hA, const void* hL,
                     const rnnt_params* pr, const int32_t* labels, const int32_t* T_len,
                     const int32_t* U_len, const float* grad_loss, void* saved, void* dhA,
                     void* dhL, float* dWA, float* dWL, float* dbZ, float* dWO, float* dbO,
                     void* ws, size_t ws_bytes, rnnt_stream stream, bool z_resident,
                     const rnnt_bwd_opts* opts = nullptr);

}  // namespace rnnt
