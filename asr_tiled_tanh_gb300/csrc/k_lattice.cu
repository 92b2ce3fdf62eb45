// k_lattice.cu -- lattice bookkeeping and the transducer loss recursion.
//
// f^W_2 / f^W_3 of "Neural transducer training: reduced memory consumption
// with sample-wise computation" (§2, Eq. 8-9): the forward variables alpha
// and backward variables beta over each sample's [T_b, U_b+1] lattice, built
// from the blank and label log-probabilities saved by the forward kernels,
// and the per-sample loss -ln P(y_b|x_b).
//
// The recursion is walked along anti-diagonals d = t + u: every position of
// a diagonal depends only on the previous diagonal, so one warp advances the
// whole front of a sample at once, each lane owning the label positions
// u = lane + 32 j.  The value handed from position u-1 (alpha) or u+1 (beta)
// moves by warp shuffles.  The log-probabilities of the diagonals ahead are
// prefetched into a register ring so the front never waits on a global load.
#include <algorithm>
#include <atomic>

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

__global__ void k_fill_f32x4(float4* __restrict__ p, float v, size_t n4) {
  const float4 q = make_float4(v, v, v, v);
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n4; i += stride) p[i] = q;
}

cudaError_t launch_fill_f32(float* p, float v, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (((uintptr_t)p & 15) != 0) {  // unaligned: one float per store
    k_fill_f32<<<grid_for(n, 256), 256, 0, s>>>(p, v, n);
    return cudaGetLastError();
  }
  const size_t n4 = n / 4, tail = n % 4;
  if (n4) k_fill_f32x4<<<grid_for(n4, 256), 256, 0, s>>>((float4*)p, v, n4);
  if (tail) k_fill_f32<<<1, 32, 0, s>>>(p + 4 * n4, v, tail);
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

__global__ void k_zero_many(ZeroList z) {
  const int i = blockIdx.y;
  unsigned char* p = (unsigned char*)z.p[i];
  const size_t n16 = z.bytes[i] / 16;
  size_t k = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; k < n16; k += stride) ((uint4*)p)[k] = make_uint4(0, 0, 0, 0);
  if (blockIdx.x == 0 && threadIdx.x < z.bytes[i] % 16) p[n16 * 16 + threadIdx.x] = 0;
}

cudaError_t launch_zero_many(const ZeroList& z, cudaStream_t s) {
  ZeroList c{};
  size_t biggest = 0;
  for (int i = 0; i < z.n && i < 8; ++i) {
    if (!z.p[i] || !z.bytes[i]) continue;
    if (((uintptr_t)z.p[i] & 15) != 0) {
      cudaError_t e = launch_zero(z.p[i], z.bytes[i], s);
      if (e != cudaSuccess) return e;
      continue;
    }
    c.p[c.n] = z.p[i];
    c.bytes[c.n] = z.bytes[i];
    biggest = biggest > z.bytes[i] ? biggest : z.bytes[i];
    ++c.n;
  }
  if (c.n == 0) return cudaSuccess;
  k_zero_many<<<dim3(grid_for(biggest / 16 + 1, 256), c.n), 256, 0, s>>>(c);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Validation + per-sample tile counts + exclusive prefix sum (one block).
// A sample is rejected (0 tiles, loss NaN) when T_len is outside [1,T],
// U_len outside [0,U1-1], or one of its labels labels[b,1..U_len] is outside
// [0,V).  labels[b,0] (the prepended blank) is never read.
constexpr int IDX_THREADS = 1024;

// Validation bits of sample b's lengths (0 if they are in range).
__device__ __forceinline__ int length_bits(const Shape& sh, int Tb, int Ub) {
  return (Tb < 1 || Tb > sh.T || Ub < 0 || Ub > sh.U1 - 1) ? status_bit(RNNT_ERR_LENGTH_RANGE)
                                                              : 0;
}

// One block.  prefix[] first holds each sample's validation bits, then its
// tile count, then its exclusive prefix: (1) lengths, one thread per sample;
// (2) every label of every sample with valid lengths, all threads over the
// flattened [B, U+1] array (coalesced; a bad label ORs a bit into its
// sample's word); (3) tile counts (0 for a rejected sample, whose loss and
// ln P become NaN); (4) block scan.
__global__ void __launch_bounds__(IDX_THREADS)
k_index(Shape sh, const int32_t* __restrict__ labels, const int32_t* __restrict__ T_len,
        const int32_t* __restrict__ U_len, SavedView sv, float* __restrict__ loss) {
  __shared__ int warp_sum[IDX_THREADS / 32];
  __shared__ int bad_bits;
  const int B = sh.B, U1 = sh.U1;
  if (threadIdx.x == 0) bad_bits = 0;
  for (int b = threadIdx.x; b < B; b += IDX_THREADS)
    sv.prefix[b] = length_bits(sh, T_len[b], U_len[b]);
  __syncthreads();
  const long long nl = (long long)B * U1;
  for (long long i = threadIdx.x; i < nl; i += IDX_THREADS) {
    const int b = (int)(i / U1), u = (int)(i % U1);
    if (u == 0 || u > U_len[b]) continue;  // the prepended blank, or past U_b
    const int y = __ldg(labels + i);
    if ((y < 0) | (y >= sh.V)) atomicOr(&sv.prefix[b], status_bit(RNNT_ERR_LABEL_RANGE));
  }
  __syncthreads();
  const int per = (int)cdiv(B, IDX_THREADS);
  const int b0 = min(B, (int)threadIdx.x * per), b1 = min(B, b0 + per);
  int local = 0, bad = 0;
  for (int b = b0; b < b1; ++b) {
    const int bits = sv.prefix[b];
    int n = 0;
    if (bits) {
      bad |= bits;
      loss[b] = NAN;
      sv.lnP[b] = NAN;
    } else {
      n = (int)(cdiv(T_len[b], TT) * cdiv(U_len[b] + 1, TU));
    }
    sv.prefix[b] = n;
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
  for (int b = b0; b < b1; ++b) {
    const int n = sv.prefix[b];
    sv.prefix[b] = run;
    run += n;
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

// One block per sample: tile j of sample b (row-major over its t and u blocks)
// is entry prefix[b] + j of the table.
__global__ void k_tile_table(Shape sh, const int32_t* __restrict__ T_len,
                             const int32_t* __restrict__ U_len, SavedView sv) {
  const int b = blockIdx.x;
  const int first = sv.prefix[b], n = sv.prefix[b + 1] - first;
  if (n <= 0) return;
  const int Tb = T_len[b], Ub = U_len[b];
  const int ntu = (int)cdiv(Ub + 1, TU);
  for (int j = threadIdx.x; j < n; j += blockDim.x)
    sv.tiles[first + j] = make_int4(b, (j / ntu) * TT, (j % ntu) * TU, Tb | (Ub << 16));
}

cudaError_t launch_tile_table(const Shape& sh, const int32_t* T_len, const int32_t* U_len,
                              SavedView sv, cudaStream_t s) {
  if (sh.B == 0) return cudaSuccess;
  k_tile_table<<<sh.B, 128, 0, s>>>(sh, T_len, U_len, sv);
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
// alpha (warp 0) and beta (warp 1) of sample blockIdx.x, one warp each.
// Lane l owns label positions u = l + 32 j (j < NJ).  Step s walks diagonal
// d = s (alpha) or d = T_b + U_b - 1 - s (beta); position (d - u, u).
//   alpha(t,u) = logaddexp(alpha(t-1,u) + lpb(t-1,u), alpha(t,u-1) + lpl(t,u-1))
//   beta(t,u)  = logaddexp(beta(t+1,u) + lpb(t,u),    beta(t,u+1) + lpl(t,u))
// with alpha(0,0) = 0, beta(T_b,U_b) := 0 (the final blank leaves the lattice)
// and -inf everywhere else outside the lattice.  Every value a position needs
// from a neighbour comes from the previous diagonal, so one diagonal is one
// round of warp shuffles (no block barrier).  The log-probabilities of the PF
// diagonals ahead sit in a register ring.
template <bool FAST>
__device__ __forceinline__ float lae(float a, float b) {
  // branch-free: when both are -inf, d = -inf and the result is m = -inf
  const float m = fmaxf(a, b);
  const float d = (m == -INFINITY) ? -INFINITY : fminf(a, b) - m;
  if (FAST) {
    // ln(1 + e^d) = ln2 * log2(1 + 2^(d log2 e))
    float e, l;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(d * 1.4426950408889634f));
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l) : "f"(1.f + e));
    return m + 0.6931471805599453f * l;
  }
  return m + log1pf(expf(d));
}

// log-add-exp of the shared-memory kernel: on the fast path its arguments
// are base-2 logarithms (both -inf: min - max is NaN, clamped to -126, and
// the result is max = -inf).
template <bool FAST>
__device__ __forceinline__ float lae_k(float a, float b) {
  if (FAST) {
    const float m = fmaxf(a, b);
    const float d = fmaxf(fminf(a, b) - m, -126.f);
    float e, l;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(d));
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l) : "f"(1.f + e));
    return m + l;
  }
  return lae<false>(a, b);
}

template <int NJ, int PF, bool FAST>
__global__ void __launch_bounds__(64)
k_alpha_beta(Shape sh, const int32_t* __restrict__ T_len, const int32_t* __restrict__ U_len,
             SavedView sv, float* __restrict__ loss) {
  const int b = blockIdx.x;
  const bool is_beta = threadIdx.x >= 32;
  const int lane = threadIdx.x & 31;
  if (sv.prefix[b + 1] == sv.prefix[b]) return;  // rejected sample: stays -inf / NaN
  const int Tb = T_len[b], Ub = U_len[b];
  const int U1 = sh.U1;
  const size_t base = (size_t)b * sh.T * U1;
  const float* __restrict__ LPB = sv.lpb + base;
  const float* __restrict__ LPL = sv.lpl + base;
  float* __restrict__ OUT = (is_beta ? sv.beta : sv.alpha) + base;
  const int ndiag = Tb + Ub;

  float rb[PF][NJ], rl[PF][NJ];
  // The ring holds raw loads from clamped (always valid) addresses; positions
  // outside the lattice are masked where the values are used, so no
  // instruction waits on a load before its diagonal comes up.
#pragma unroll
  for (int k = 0; k < PF; ++k) {
    const int d = is_beta ? ndiag - 1 - k : k;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int u = min(lane + 32 * j, Ub), t = min(max(d - (lane + 32 * j), 0), Tb - 1);
      rb[k][j] = LPB[(size_t)t * U1 + u];
      rl[k][j] = LPL[(size_t)t * U1 + u];
    }
  }
  float own[NJ], send[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) own[j] = send[j] = -INFINITY;

  for (int sb = 0; sb < ndiag; sb += PF) {
#pragma unroll
    for (int k = 0; k < PF; ++k) {
      const int s = sb + k;
      if (s < ndiag) {  // uniform over the warp
        const int d = is_beta ? ndiag - 1 - s : s;
        float nb[NJ];
        // neighbour values from the previous diagonal
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          if (!is_beta) {
            float x = __shfl_up_sync(0xffffffffu, send[j], 1);
            const float y = __shfl_sync(0xffffffffu, j > 0 ? send[j - 1] : -INFINITY, 31);
            nb[j] = lane == 0 ? y : x;
          } else {
            float x = __shfl_down_sync(0xffffffffu, send[j], 1);
            const float y = __shfl_sync(0xffffffffu, j + 1 < NJ ? send[j + 1] : -INFINITY, 0);
            nb[j] = lane == 31 ? y : x;
          }
        }
        const int s2 = s + PF;
        const int d2 = is_beta ? ndiag - 1 - s2 : s2;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int u = lane + 32 * j, t = d - u;
          const bool in = u <= Ub && t >= 0 && t < Tb;
          const float lb = in ? rb[k][j] : -INFINITY;
          const float ll = in ? rl[k][j] : -INFINITY;
          {
            const int uc = min(u, Ub), t2 = min(max(d2 - u, 0), Tb - 1);
            rb[k][j] = LPB[(size_t)t2 * U1 + uc];
            rl[k][j] = LPL[(size_t)t2 * U1 + uc];
          }
          float val = -INFINITY;
          if (in) {
            if (!is_beta) {
              val = (s == 0) ? 0.f : lae<FAST>(own[j], nb[j]);
            } else {
              const float from_t = (t + 1 < Tb) ? own[j] : (u == Ub ? 0.f : -INFINITY);
              val = lae<FAST>(from_t + lb, nb[j] + ll);
            }
            OUT[(size_t)t * U1 + u] = val;
          }
          if (!is_beta) {
            own[j] = val + lb;   // alpha + lpb: the blank move to (t+1, u)
            send[j] = val + ll;  // alpha + lpl: the label move to (t, u+1)
          } else {
            own[j] = val;
            send[j] = val;
          }
        }
      }
    }
  }
  // ln P = alpha(T_b-1, U_b) + lpb(T_b-1, U_b): the own value at u = U_b
  // after the last diagonal.
  if (!is_beta) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (lane + 32 * j == Ub) {
        sv.lnP[b] = own[j];
        loss[b] = -own[j];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The same recursion with the log-probabilities streamed through shared
// memory: rows of the sample's lattice are copied (cp.async) in windows of 32
// rows into a circular buffer of R rows (R a power of two, at least
// ceil(U1/32) + 2 windows), one window ahead of the wavefront, so the diagonal
// loop reads only shared memory.  The front at diagonal d spans rows
// [max(0, d - U_b), min(d, T_b - 1)], at most ceil(U1/32) + 1 windows.
// Lane l owns the NJ consecutive label positions u = NJ*l + j, so a diagonal
// needs a single shuffle (for j = 0 with alpha, j = NJ-1 with beta).
// One warp per block: alpha (blockIdx.y == 0) or beta (blockIdx.y == 1).
constexpr int AB_W = 32;

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One direction of the recursion for one sample (one warp).  The per-lane
// state advances by increments from one diagonal to the next: position j's
// frame t, its row in the ring and its offset in the output array.
template <int NJ, bool FAST, bool BETA, int W>
__device__ __forceinline__ void ab_walk(float* ring, float* xch, int R, int Tb, int Ub, int U1,
                                        const float* __restrict__ LPB,
                                        const float* __restrict__ LPL, float* __restrict__ OUT,
                                        float* lnP, float* loss) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int plane = R * U1;
  const int rmask = R - 1;
  const int nwin = (Tb + AB_W - 1) / AB_W;
  const int ndiag = Tb + Ub;
  // The fast path runs the recursion on base-2 logarithms: inputs are scaled
  // by log2 e as they are read, results by ln 2 as they are stored, so the
  // log-add-exp on the dependency chain is max + lg2(1 + 2^(min - max)).
  constexpr float kIn = FAST ? 1.4426950408889634f : 1.f;
  constexpr float kOut = FAST ? 0.6931471805599453f : 1.f;

  auto load_window = [&](int w) {  // rows [w*32, w*32+32) of lpb and lpl
    const int r0 = w * AB_W, r1 = min(Tb, r0 + AB_W);
    const int n = (r1 - r0) * U1;
    float* dst = ring + (r0 & rmask) * U1;
    const float* gb = LPB + (size_t)r0 * U1;
    const float* gl = LPL + (size_t)r0 * U1;
    for (int i = threadIdx.x; i < n; i += 32 * W) {
      cp_async4(dst + i, gb + i);
      cp_async4(dst + plane + i, gl + i);
    }
    cp_async_commit();
  };
  // every thread's copies of a window are complete, and seen by all warps
  auto window_sync = [&]() {
    cp_async_wait<1>();
    if (W > 1) __syncthreads(); else __syncwarp();
  };
  int next_win, ready;  // next window to load; window known complete
  if (!BETA) {
    load_window(0);
    if (nwin > 1) load_window(1); else cp_async_commit();
    next_win = 2;
    ready = 0;
  } else {
    load_window(nwin - 1);
    if (nwin > 1) load_window(nwin - 2); else cp_async_commit();
    next_win = nwin - 3;
    ready = nwin - 1;
  }
  window_sync();

  const int u0 = NJ * (warp * 32 + lane);
  const int d0 = BETA ? ndiag - 1 : 0;
  int t[NJ], ri[NJ], oo[NJ];
  bool uok[NJ], ulast[NJ];
  float own[NJ], send[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int u = u0 + j;
    uok[j] = u <= Ub;
    ulast[j] = u == Ub;
    t[j] = d0 - u;
    ri[j] = (t[j] & rmask) * U1 + min(u, U1 - 1);  // always inside the ring
    oo[j] = t[j] * U1 + u;
    own[j] = send[j] = -INFINITY;
  }

#pragma unroll 2
  for (int s = 0; s < ndiag; ++s) {
    const int d = BETA ? ndiag - 1 - s : s;
    if (!BETA) {
      const int hi = min(d, Tb - 1) >> 5;
      if (hi > ready) {  // entering window `hi`, loaded one ahead
        if (next_win < nwin) { load_window(next_win); ++next_win; } else cp_async_commit();
        window_sync();
        ready = hi;
      }
    } else {
      const int lo = max(0, d - Ub) >> 5;
      if (lo < ready) {
        if (next_win >= 0) { load_window(next_win); --next_win; } else cp_async_commit();
        window_sync();
        ready = lo;
      }
    }
    // neighbours from the previous diagonal: a shuffle within the warp, the
    // neighbouring warp's edge value through shared memory (written at the
    // end of the previous diagonal, before the barrier)
    float nb[NJ];
    const float* xin = xch + ((s + 1) & 1) * W;
    if (!BETA) {
      const float x = __shfl_up_sync(0xffffffffu, send[NJ - 1], 1);
      nb[0] = lane > 0 ? x : ((W > 1 && warp > 0 && s > 0) ? xin[warp - 1] : -INFINITY);
#pragma unroll
      for (int j = 1; j < NJ; ++j) nb[j] = send[j - 1];
    } else {
      const float x = __shfl_down_sync(0xffffffffu, send[0], 1);
      nb[NJ - 1] = lane < 31 ? x : ((W > 1 && warp < W - 1 && s > 0) ? xin[warp + 1] : -INFINITY);
#pragma unroll
      for (int j = 0; j < NJ - 1; ++j) nb[j] = send[j + 1];
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const bool in = uok[j] && (unsigned)t[j] < (unsigned)Tb;
      const float lb = in ? ring[ri[j]] * kIn : -INFINITY;
      const float ll = in ? ring[ri[j] + plane] * kIn : -INFINITY;
      float val;
      if (!BETA) {
        val = (s == 0) ? 0.f : lae_k<FAST>(own[j], nb[j]);
      } else {
        const float from_t = (t[j] + 1 < Tb) ? own[j] : (ulast[j] ? 0.f : -INFINITY);
        val = lae_k<FAST>(from_t + lb, nb[j] + ll);
      }
      val = in ? val : -INFINITY;
      if (in) OUT[oo[j]] = val * kOut;
      if (!BETA) {
        own[j] = val + lb;   // alpha + lpb: the blank move to (t+1, u)
        send[j] = val + ll;  // alpha + lpl: the label move to (t, u+1)
        ++t[j];
        ri[j] += U1;
        if (ri[j] >= plane) ri[j] -= plane;
        oo[j] += U1;
      } else {
        own[j] = val;
        send[j] = val;
        --t[j];
        ri[j] -= U1;
        if (ri[j] < 0) ri[j] += plane;
        oo[j] -= U1;
      }
    }
    if (W > 1) {
      // the warp's edge value for its neighbour warp on the next diagonal
      float* xout = xch + (s & 1) * W;
      if (!BETA && lane == 31) xout[warp] = send[NJ - 1];
      if (BETA && lane == 0) xout[warp] = send[0];
      __syncthreads();
    }
  }
  cp_async_wait<0>();
  if (!BETA) {
    // ln P = alpha(T_b-1, U_b) + lpb(T_b-1, U_b): the own value at u = U_b
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (ulast[j]) {
        *lnP = own[j] * kOut;
        *loss = -own[j] * kOut;
      }
    }
  }
}

// W warps per block split the label positions of one sample (lane l of warp
// w owns u = NJ (32 w + l) ..); with W > 1 the warps meet at a barrier once
// per diagonal.  Several warps pay off when there are few samples (the
// recursion is latency-bound, and the GPU otherwise runs 2B warps).
// ---------------------------------------------------------------------------
// The recursion for batches whose walks outnumber the SMs: instead of whole
// rows (the ring above needs room for U1 + 64 rows of the lattice, one walk
// per SM at U1 = 101), a walk keeps only the next KD diagonals of its
// sample's log-probabilities in shared memory, double-buffered: two bands of
// KD x 32 NJ entries per array.  A band is filled by cp.async from row
// segments: for row t the diagonals d0 .. d0+KD-1 of the band hold KD
// consecutive label positions u = d - t, so the lanes of a warp copy 32/KD
// contiguous row pieces per instruction (the register-prefetch walk reads 32
// rows per instruction).  Entry (d, u) sits at [d - d0][u % NJ][u / NJ], so
// that the lanes, which own u = NJ lane + j, read consecutive words.
constexpr int AB_KD = 8;  // diagonals per band

template <int NJ, bool FAST, bool BETA>
__device__ __forceinline__ void ab_walk_band(float* band, int Tb, int Ub, int U1,
                                             const float* __restrict__ LPB,
                                             const float* __restrict__ LPL,
                                             float* __restrict__ OUT, float* lnP, float* loss) {
  constexpr int KD = AB_KD, UP = 32 * NJ, BAND = KD * UP;
  const int lane = threadIdx.x & 31;
  const int ndiag = Tb + Ub;
  const int nband = (ndiag + KD - 1) / KD;
  constexpr float kIn = FAST ? 1.4426950408889634f : 1.f;
  constexpr float kOut = FAST ? 0.6931471805599453f : 1.f;
  // band b holds walk steps s in [b KD, b KD + KD): diagonals from its lowest
  // one, dlo(b) (alpha: d = s; beta: d = ndiag - 1 - s), possibly below 0
  auto band_lo = [&](int b) { return BETA ? ndiag - (b + 1) * KD : b * KD; };
  auto load_band = [&](int b) {
    float* dst = band + (b & 1) * 2 * BAND;  // the band's lpb entries, then its lpl ones
    const int d0 = band_lo(b);
    const int t0 = max(0, d0 - Ub), t1 = min(Tb - 1, d0 + KD - 1);
    const int n = (t1 - t0 + 1) * KD;
    for (int i = lane; i < n; i += 32) {
      const int t = t0 + i / KD, c = i % KD, d = d0 + c, u = d - t;
      if (d >= 0 && d < ndiag && u >= 0 && u <= Ub) {
        const int k = c * UP + (u % NJ) * 32 + u / NJ;
        cp_async4(dst + k, LPB + (size_t)t * U1 + u);
        cp_async4(dst + BAND + k, LPL + (size_t)t * U1 + u);
      }
    }
    cp_async_commit();
  };
  load_band(0);
  if (nband > 1) load_band(1); else cp_async_commit();
  cp_async_wait<1>();
  __syncwarp();

  const int u0 = NJ * lane;
  const int d0 = BETA ? ndiag - 1 : 0;
  int t[NJ], oo[NJ];
  bool uok[NJ], ulast[NJ];
  float own[NJ], send[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int u = u0 + j;
    uok[j] = u <= Ub;
    ulast[j] = u == Ub;
    t[j] = d0 - u;
    oo[j] = t[j] * U1 + u;
    own[j] = send[j] = -INFINITY;
  }

  for (int s = 0; s < ndiag; ++s) {
    const int b = s / KD, c = s - b * KD;
    if (c == 0 && b > 0) {
      // entering band b: every lane is done with band b-1, whose buffer takes
      // band b+1; band b (issued one band ago) is complete after the wait
      __syncwarp();
      if (b + 1 < nband) load_band(b + 1); else cp_async_commit();
      cp_async_wait<1>();
      __syncwarp();
    }
    const float* cur = band + (b & 1) * 2 * BAND + (BETA ? KD - 1 - c : c) * UP + lane;
    float nb[NJ];
    if (!BETA) {
      const float x = __shfl_up_sync(0xffffffffu, send[NJ - 1], 1);
      nb[0] = lane > 0 ? x : -INFINITY;
#pragma unroll
      for (int j = 1; j < NJ; ++j) nb[j] = send[j - 1];
    } else {
      const float x = __shfl_down_sync(0xffffffffu, send[0], 1);
      nb[NJ - 1] = lane < 31 ? x : -INFINITY;
#pragma unroll
      for (int j = 0; j < NJ - 1; ++j) nb[j] = send[j + 1];
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const bool in = uok[j] && (unsigned)t[j] < (unsigned)Tb;
      const float lb = in ? cur[j * 32] * kIn : -INFINITY;
      const float ll = in ? cur[BAND + j * 32] * kIn : -INFINITY;
      float val;
      if (!BETA) {
        val = (s == 0) ? 0.f : lae_k<FAST>(own[j], nb[j]);
      } else {
        const float from_t = (t[j] + 1 < Tb) ? own[j] : (ulast[j] ? 0.f : -INFINITY);
        val = lae_k<FAST>(from_t + lb, nb[j] + ll);
      }
      val = in ? val : -INFINITY;
      if (in) OUT[oo[j]] = val * kOut;
      if (!BETA) {
        own[j] = val + lb;   // alpha + lpb: the blank move to (t+1, u)
        send[j] = val + ll;  // alpha + lpl: the label move to (t, u+1)
        ++t[j];
        oo[j] += U1;
      } else {
        own[j] = val;
        send[j] = val;
        --t[j];
        oo[j] -= U1;
      }
    }
  }
  cp_async_wait<0>();
  if (!BETA) {
    // ln P = alpha(T_b-1, U_b) + lpb(T_b-1, U_b): the own value at u = U_b
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (ulast[j]) {
        *lnP = own[j] * kOut;
        *loss = -own[j] * kOut;
      }
    }
  }
}

template <int NJ, bool FAST>
__global__ void __launch_bounds__(32)
k_alpha_beta_band(Shape sh, const int32_t* __restrict__ T_len, const int32_t* __restrict__ U_len,
                  SavedView sv, float* __restrict__ loss) {
  __shared__ float band[2 * 2 * AB_KD * 32 * NJ];
  const int b = blockIdx.x;
  if (sv.prefix[b + 1] == sv.prefix[b]) return;  // rejected sample
  const int Tb = T_len[b], Ub = U_len[b];
  const size_t base = (size_t)b * sh.T * sh.U1;
  if (blockIdx.y == 0)
    ab_walk_band<NJ, FAST, false>(band, Tb, Ub, sh.U1, sv.lpb + base, sv.lpl + base,
                                  sv.alpha + base, sv.lnP + b, loss + b);
  else
    ab_walk_band<NJ, FAST, true>(band, Tb, Ub, sh.U1, sv.lpb + base, sv.lpl + base,
                                 sv.beta + base, nullptr, nullptr);
}

template <bool FAST>
static cudaError_t launch_ab_band(const Shape& sh, const int32_t* T_len, const int32_t* U_len,
                                  SavedView sv, float* loss, cudaStream_t s) {
  const int nj = (int)cdiv(sh.U1, 32);
  const dim3 g(sh.B, 2);
  if (nj <= 1) k_alpha_beta_band<1, FAST><<<g, 32, 0, s>>>(sh, T_len, U_len, sv, loss);
  else if (nj <= 2) k_alpha_beta_band<2, FAST><<<g, 32, 0, s>>>(sh, T_len, U_len, sv, loss);
  else k_alpha_beta_band<4, FAST><<<g, 32, 0, s>>>(sh, T_len, U_len, sv, loss);
  return cudaGetLastError();
}

template <int NJ, bool FAST, int W>
__global__ void __launch_bounds__(32 * W)
k_alpha_beta_smem(Shape sh, const int32_t* __restrict__ T_len, const int32_t* __restrict__ U_len,
                  SavedView sv, float* __restrict__ loss, int R) {
  extern __shared__ float ring[];  // [lpb | lpl] x R rows x U1, then 2 x W exchange slots
  float* xch = ring + 2 * (size_t)R * sh.U1;
  const int b = blockIdx.x;
  if (sv.prefix[b + 1] == sv.prefix[b]) return;  // rejected sample (uniform over the block)
  const int Tb = T_len[b], Ub = U_len[b];
  const size_t base = (size_t)b * sh.T * sh.U1;
  if (blockIdx.y == 0)
    ab_walk<NJ, FAST, false, W>(ring, xch, R, Tb, Ub, sh.U1, sv.lpb + base, sv.lpl + base,
                                sv.alpha + base, sv.lnP + b, loss + b);
  else
    ab_walk<NJ, FAST, true, W>(ring, xch, R, Tb, Ub, sh.U1, sv.lpb + base, sv.lpl + base,
                               sv.beta + base, nullptr, nullptr);
}

template <bool FAST>
static cudaError_t launch_ab(const Shape& sh, const int32_t* T_len, const int32_t* U_len,
                             SavedView sv, float* loss, cudaStream_t s) {
  const int nj = (int)cdiv(sh.U1, 32);
  dim3 g(sh.B), blk(64);
  if (nj <= 1) k_alpha_beta<1, 16, FAST><<<g, blk, 0, s>>>(sh, T_len, U_len, sv, loss);
  else if (nj <= 2) k_alpha_beta<2, 16, FAST><<<g, blk, 0, s>>>(sh, T_len, U_len, sv, loss);
  else if (nj <= 4) k_alpha_beta<4, 12, FAST><<<g, blk, 0, s>>>(sh, T_len, U_len, sv, loss);
  else if (nj <= 8) k_alpha_beta<8, 6, FAST><<<g, blk, 0, s>>>(sh, T_len, U_len, sv, loss);
  else if (nj <= 16) k_alpha_beta<16, 3, FAST><<<g, blk, 0, s>>>(sh, T_len, U_len, sv, loss);
  else k_alpha_beta<32, 1, FAST><<<g, blk, 0, s>>>(sh, T_len, U_len, sv, loss);
  return cudaGetLastError();
}

template <int NJ, bool FAST, int W>
static cudaError_t launch_ab_smem(const Shape& sh, const int32_t* T_len, const int32_t* U_len,
                                  SavedView sv, float* loss, int R, size_t smem,
                                  cudaStream_t s) {
  static std::atomic<bool> attr[kDeviceSlots];  // per instantiation and device
  std::atomic<bool>& done = attr[device_slot()];
  if (!done.load()) {
    cudaError_t e = cudaFuncSetAttribute(k_alpha_beta_smem<NJ, FAST, W>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    if (e != cudaSuccess) return e;
    done.store(true);
  }
  k_alpha_beta_smem<NJ, FAST, W><<<dim3(sh.B, 2), 32 * W, smem, s>>>(sh, T_len, U_len, sv, loss,
                                                                       R);
  return cudaGetLastError();
}

int num_sms() {
  static std::atomic<int> count[kDeviceSlots];
  std::atomic<int>& cached = count[device_slot()];
  int n = cached.load();
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();  // (no device: clear the error state)
      n = 152;
    }
    cached.store(n);
  }
  return n;
}

template <bool FAST>
static cudaError_t launch_ab_smem_nj(const Shape& sh, const int32_t* T_len, const int32_t* U_len,
                                     SavedView sv, float* loss, int R, size_t smem, int w,
                                     cudaStream_t s) {
  const int nj = (int)cdiv(sh.U1, 32 * w);
  if (w == 4) return launch_ab_smem<1, FAST, 4>(sh, T_len, U_len, sv, loss, R, smem, s);
  if (w == 2) {
    if (nj <= 1) return launch_ab_smem<1, FAST, 2>(sh, T_len, U_len, sv, loss, R, smem, s);
    return launch_ab_smem<2, FAST, 2>(sh, T_len, U_len, sv, loss, R, smem, s);
  }
  if (nj <= 1) return launch_ab_smem<1, FAST, 1>(sh, T_len, U_len, sv, loss, R, smem, s);
  if (nj <= 2) return launch_ab_smem<2, FAST, 1>(sh, T_len, U_len, sv, loss, R, smem, s);
  return launch_ab_smem<4, FAST, 1>(sh, T_len, U_len, sv, loss, R, smem, s);
}

cudaError_t launch_alpha_beta(const Shape& sh, const int32_t* T_len, const int32_t* U_len,
                              SavedView sv, float* loss, bool fast, cudaStream_t s) {
  if (sh.B == 0) return cudaSuccess;
  if (sh.U1 > 1024) return cudaErrorInvalidValue;
  // shared-memory ring when it fits in 220 KiB and the 2B walks it leaves
  // resident finish in at most two waves; more walks take the band kernel
  // (16 KiB per walk, every walk resident at once: at B=1024, U=100 the ring
  // allows one walk per SM, 13.5 waves), or the register-prefetch kernel when
  // U1 > 128
  int R = AB_W;
  while (R < ((int)cdiv(sh.U1, AB_W) + 2) * AB_W) R *= 2;
  const size_t smem = (size_t)2 * R * sh.U1 * sizeof(float) + 2 * 4 * sizeof(float);
  const int nj = (int)cdiv(sh.U1, 32);
  const long long per_sm = std::max<long long>(1, (228LL * 1024) / (long long)(smem + 1024));
  const bool few_waves = 2LL * sh.B <= 2LL * per_sm * num_sms();
  if (smem <= 220 * 1024 && nj <= 4 && few_waves) {
    // warps per sample and direction: one label position per lane when the
    // 2B recursions leave most SMs idle, else one warp (several positions each)
    int w = 1;
    if (nj > 1 && 2LL * sh.B * nj <= 2LL * num_sms()) w = nj <= 2 ? 2 : 4;
    return fast ? launch_ab_smem_nj<true>(sh, T_len, U_len, sv, loss, R, smem, w, s)
                : launch_ab_smem_nj<false>(sh, T_len, U_len, sv, loss, R, smem, w, s);
  }
  if (nj <= 4)
    return fast ? launch_ab_band<true>(sh, T_len, U_len, sv, loss, s)
                : launch_ab_band<false>(sh, T_len, U_len, sv, loss, s);
  return fast ? launch_ab<true>(sh, T_len, U_len, sv, loss, s)
              : launch_ab<false>(sh, T_len, U_len, sv, loss, s);
}

}  // namespace rnnt
