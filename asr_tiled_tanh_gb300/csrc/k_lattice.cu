// k_lattice.cu -- lattice bookkeeping and the transducer loss recursion.
//
// f^W_2 / f^W_3 of "Neural transducer training: reduced memory consumption
// with sample-wise computation" (§2, Eq. 8-9): the forward variables alpha
// and backward variables beta over each sample's [T_b, U_b+1] lattice, built
// from the blank and label log-probabilities saved by the forward kernels,
// and the per-sample loss -ln P(y_b|x_b).
//
// The recursion is walked along anti-diagonals d = t + u: every position of
// a diagonal depends only on the previous diagonal, so one thread per label
// position u advances the whole front at once.  The value handed from
// position u-1 (alpha) or u+1 (beta) moves by a warp shuffle, and across warp
// boundaries through a double-buffered shared-memory slot with one barrier
// per diagonal.  The log-probabilities of the diagonals ahead are prefetched
// into a register ring so the front never waits on a global load.
#include "kernels.h"

namespace rnnt {

__global__ void k_fill_f32(float* __restrict__ p, float v, size_t n) {
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n; i += stride) p[i] = v;
}

__global__ void k_zero16(uint4* __restrict__ p, size_t n16) {
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n16; i += stride) p[i] = make_uint4(0, 0, 0, 0);
}

__global__ void k_zero1(unsigned char* __restrict__ p, size_t n) {
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0;
}

static int grid_for(size_t n, int threads) {
  size_t g = (n + threads - 1) / threads;
  if (g > 152 * 32) g = 152 * 32;
  return g < 1 ? 1 : (int)g;
}

cudaError_t launch_fill_f32(float* p, float v, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  k_fill_f32<<<grid_for(n, 256), 256, 0, s>>>(p, v, n);
  return cudaGetLastError();
}

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  size_t n16 = bytes / 16, tail = bytes % 16;
  if (((uintptr_t)p & 15) != 0) {  // unaligned: byte kernel
    k_zero1<<<(unsigned)((bytes + 255) / 256), 256, 0, s>>>((unsigned char*)p, bytes);
    return cudaGetLastError();
  }
  if (n16) k_zero16<<<grid_for(n16, 256), 256, 0, s>>>((uint4*)p, n16);
  if (tail) k_zero1<<<1, 32, 0, s>>>((unsigned char*)p + n16 * 16, tail);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Validation + per-sample tile counts + exclusive prefix sum (one block).
// A sample is rejected (0 tiles, loss NaN) when T_len is outside [1,T],
// U_len outside [0,U1-1], or one of its labels labels[b,1..U_len] is outside
// [0,V).  labels[b,0] (the prepended blank) is never read.
constexpr int IDX_THREADS = 1024;

// Tiles of sample b, or 0 (and a status bit in *bad) if it is rejected.
__device__ inline int sample_tiles(const Shape& sh, const int32_t* __restrict__ labels,
                                   const int32_t* __restrict__ T_len,
                                   const int32_t* __restrict__ U_len, int b, int* bad) {
  const int Tb = T_len[b], Ub = U_len[b];
  if (Tb < 1 || Tb > sh.T || Ub < 0 || Ub > sh.U1 - 1) {
    *bad |= status_bit(RNNT_ERR_LENGTH_RANGE);
    return 0;
  }
  const int32_t* lab = labels + (size_t)b * sh.U1;
  for (int u = 1; u <= Ub; ++u) {
    const int y = lab[u];
    if (y < 0 || y >= sh.V) {
      *bad |= status_bit(RNNT_ERR_LABEL_RANGE);
      return 0;
    }
  }
  return (int)(cdiv(Tb, TT) * cdiv(Ub + 1, TU));
}

__global__ void __launch_bounds__(IDX_THREADS)
k_index(Shape sh, const int32_t* __restrict__ labels, const int32_t* __restrict__ T_len,
        const int32_t* __restrict__ U_len, SavedView sv, float* __restrict__ loss) {
  __shared__ int warp_sum[IDX_THREADS / 32];
  __shared__ int bad_bits;
  const int B = sh.B;
  const int per = (int)cdiv(B, IDX_THREADS);
  const int b0 = min(B, (int)threadIdx.x * per), b1 = min(B, b0 + per);
  if (threadIdx.x == 0) bad_bits = 0;
  __syncthreads();
  int local = 0, bad = 0;
  for (int b = b0; b < b1; ++b) {
    const int n = sample_tiles(sh, labels, T_len, U_len, b, &bad);
    if (n == 0) {
      loss[b] = NAN;
      sv.lnP[b] = NAN;
    }
    local += n;
  }
  // block exclusive scan of `local`
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[w] = incl;
  if (bad) atomicOr(&bad_bits, bad);
  __syncthreads();
  if (w == 0) {
    int v = warp_sum[lane];
    int s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int x = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += x;
    }
    warp_sum[lane] = s - v;  // exclusive warp offsets
  }
  __syncthreads();
  int run = warp_sum[w] + incl - local;
  int dummy = 0;
  for (int b = b0; b < b1; ++b) {
    sv.prefix[b] = run;
    run += sample_tiles(sh, labels, T_len, U_len, b, &dummy);
  }
  if (threadIdx.x == IDX_THREADS - 1) {
    sv.prefix[B] = run;
    *sv.total_tiles = run;
    *sv.status = bad_bits;
  }
}

cudaError_t launch_index(const Shape& sh, const int32_t* labels, const int32_t* T_len,
                         const int32_t* U_len, SavedView sv, float* loss, cudaStream_t s) {
  k_index<<<1, IDX_THREADS, 0, s>>>(sh, labels, T_len, U_len, sv, loss);
  return cudaGetLastError();
}

__global__ void k_eff_lengths(int B, SavedView sv, const int32_t* __restrict__ T_len,
                              const int32_t* __restrict__ U_len, int32_t* __restrict__ Teff,
                              int32_t* __restrict__ Ueff) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const bool ok = sv.prefix[b + 1] > sv.prefix[b];
  Teff[b] = ok ? T_len[b] : 0;
  Ueff[b] = ok ? U_len[b] + 1 : 0;
}

cudaError_t launch_eff_lengths(const Shape& sh, SavedView sv, const int32_t* T_len,
                               const int32_t* U_len, int32_t* Teff, int32_t* Ueff,
                               cudaStream_t s) {
  if (sh.B == 0) return cudaSuccess;
  k_eff_lengths<<<(unsigned)cdiv(sh.B, 256), 256, 0, s>>>(sh.B, sv, T_len, U_len, Teff, Ueff);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// alpha (blockIdx.y == 0) and beta (blockIdx.y == 1) of sample blockIdx.x.
// Thread u owns label position u.  Step s walks diagonal d = s (alpha) or
// d = T_b + U_b - 1 - s (beta); the thread's position on it is (d - u, u).
//   alpha(t,u) = logaddexp(alpha(t-1,u) + lpb(t-1,u), alpha(t,u-1) + lpl(t,u-1))
//   beta(t,u)  = logaddexp(beta(t+1,u) + lpb(t,u),    beta(t,u+1) + lpl(t,u))
// with alpha(0,0) = 0, beta(T_b,U_b) := 0 (the final blank leaves the
// lattice) and -inf everywhere else outside the lattice.
constexpr int AB_PF = 8;

__global__ void k_alpha_beta(Shape sh, const int32_t* __restrict__ T_len,
                             const int32_t* __restrict__ U_len, SavedView sv,
                             float* __restrict__ loss) {
  __shared__ float xbuf[2][32];
  const int b = blockIdx.x;
  const bool is_beta = blockIdx.y != 0;
  if (sv.prefix[b + 1] == sv.prefix[b]) return;  // rejected sample: stays -inf / NaN
  const int Tb = T_len[b], Ub = U_len[b];
  const int U1 = sh.U1;
  const int u = threadIdx.x, lane = u & 31, w = u >> 5, NW = blockDim.x >> 5;
  const size_t base = (size_t)b * sh.T * U1;
  const float* __restrict__ LPB = sv.lpb + base;
  const float* __restrict__ LPL = sv.lpl + base;
  float* __restrict__ OUT = (is_beta ? sv.beta : sv.alpha) + base;
  const int ndiag = Tb + Ub;
  const bool u_ok = u <= Ub;
  if (threadIdx.x < 64) (&xbuf[0][0])[threadIdx.x] = -INFINITY;
  __syncthreads();

  float rb[AB_PF], rl[AB_PF];
#pragma unroll
  for (int k = 0; k < AB_PF; ++k) {
    const int d = is_beta ? ndiag - 1 - k : k;
    const int t = d - u;
    const bool in = k < ndiag && u_ok && t >= 0 && t < Tb;
    rb[k] = in ? LPB[(size_t)t * U1 + u] : -INFINITY;
    rl[k] = in ? LPL[(size_t)t * U1 + u] : -INFINITY;
  }
  float own = -INFINITY;   // alpha: alpha+lpb of the own position one diagonal back
                           // beta:  beta of the own position one diagonal back
  float send = -INFINITY;  // alpha: alpha+lpl handed to u+1; beta: beta handed to u-1

  for (int sb = 0; sb < ndiag; sb += AB_PF) {
#pragma unroll
    for (int k = 0; k < AB_PF; ++k) {
      const int s = sb + k;
      if (s < ndiag) {  // uniform over the block
        const int d = is_beta ? ndiag - 1 - s : s;
        const int t = d - u;
        const float lb = rb[k], ll = rl[k];
        {
          const int s2 = s + AB_PF;
          const int d2 = is_beta ? ndiag - 1 - s2 : s2;
          const int t2 = d2 - u;
          const bool in2 = s2 < ndiag && u_ok && t2 >= 0 && t2 < Tb;
          rb[k] = in2 ? LPB[(size_t)t2 * U1 + u] : -INFINITY;
          rl[k] = in2 ? LPL[(size_t)t2 * U1 + u] : -INFINITY;
        }
        float nb;
        if (!is_beta) {
          nb = __shfl_up_sync(0xffffffffu, send, 1);
          if (lane == 0) nb = (w > 0) ? xbuf[(s + 1) & 1][w - 1] : -INFINITY;
        } else {
          nb = __shfl_down_sync(0xffffffffu, send, 1);
          if (lane == 31) nb = (w < NW - 1) ? xbuf[(s + 1) & 1][w + 1] : -INFINITY;
        }
        float val = -INFINITY;
        const bool in = u_ok && t >= 0 && t < Tb;
        if (in) {
          if (!is_beta) {
            val = (s == 0) ? 0.f : logaddexp_f(own, nb);
          } else {
            const float from_t = (t + 1 < Tb) ? own : (u == Ub ? 0.f : -INFINITY);
            val = logaddexp_f(from_t + lb, nb + ll);
          }
          OUT[(size_t)t * U1 + u] = val;
        }
        if (!is_beta) {
          own = val + lb;
          send = val + ll;
        } else {
          own = val;
          send = val;
        }
        if (NW > 1) {
          if (!is_beta && lane == 31) xbuf[s & 1][w] = send;
          if (is_beta && lane == 0) xbuf[s & 1][w] = send;
          __syncthreads();
        }
      }
    }
  }
  // ln P = alpha(T_b-1, U_b) + lpb(T_b-1, U_b): the own value of thread U_b
  // after the last diagonal.
  if (!is_beta && u == Ub) {
    sv.lnP[b] = own;
    loss[b] = -own;
  }
}

cudaError_t launch_alpha_beta(const Shape& sh, const int32_t* T_len, const int32_t* U_len,
                              SavedView sv, float* loss, cudaStream_t s) {
  if (sh.B == 0) return cudaSuccess;
  const int threads = (int)cdiv(sh.U1, 32) * 32;
  k_alpha_beta<<<dim3(sh.B, 2), threads, 0, s>>>(sh, T_len, U_len, sv, loss);
  return cudaGetLastError();
}

}  // namespace rnnt
