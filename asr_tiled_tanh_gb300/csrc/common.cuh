// common.cuh -- internal plan, buffer layout and tile geometry shared by the
// kernels and the C-ABI host code of librnnt_gb300.
//
// Lattice tiles.  The Flash RNN-T blog ("Compute it, use it, make room")
// groups lattice positions into tiles and keeps the large intermediates only
// for the tiles in flight.  Here a tile is a 32 (t) x 4 (u) block of one
// sample's lattice: 128 positions, one per TMEM lane / epilogue thread in the
// tensor-core kernels.  (A sample's lattice is padded to whole tiles; with
// label lengths of tens of symbols and hundreds of frames, rounding U_b + 1
// up to 4 and T_b up to 32 wastes fewer positions than 8 and 16: 4.5%
// against 6.2% of the rows at the 40 s workload's lengths.)  Only tiles that intersect a sample's lattice exist
// (per-sample padding removal, as in the sample-wise paper's conclusion);
// positions of an edge tile that fall outside the lattice are masked.
// Tiles are numbered sample-major, then t-block, then u-block; the exclusive
// prefix sum of per-sample tile counts lives in `saved`.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <math.h>

#include "../../include/rnnt.h"

namespace rnnt {

constexpr int TT = 32;            // t extent of a tile
constexpr int TU = 4;             // u extent of a tile
constexpr int TILE = TT * TU;     // lattice positions per tile (= 128 MMA rows)
constexpr size_t ALIGN = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a = ALIGN) {
  return (x + a - 1) / a * a;
}

// Host state that a launcher sets up once per device (function attributes,
// occupancy figures, SM counts) is kept in per-device slots, so that a process
// may drive several GPUs.
constexpr int kDeviceSlots = 64;
inline int device_slot() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0) d = 0;
  return d % kDeviceSlots;
}
__host__ __device__ inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// Status word bits: bit k <=> rnnt_status k.
__host__ __device__ constexpr int status_bit(int code) { return 1 << code; }

// Everything the host derives from rnnt_dims before launching.
struct Plan {
  int B, T, U1, HA, HL, H, V, blank, dtype, mode;
  bool tc;                  // bf16 tensor-core path (else fp32 SIMT path)
  bool f8;                  // the score GEMMs on e4m3 operands (dtype RNNT_BF16_E4M3)
  long long max_tiles;      // tiles when every sample has full lengths
  long long chunk_tiles;    // tiles whose intermediates are held at once
  long long chunk_rows;     // = chunk_tiles * TILE
  int zelem, helem;         // bytes per element of the z and score buffers
  // saved layout
  size_t s_status, s_prefix, s_tiles, s_lnP, s_lpb, s_lpl, s_lnPD, s_alpha, s_beta, s_pA, s_pL, s_z, s_h,
      s_total;
  // workspace layout
  size_t w_dA, w_dLr, w_z, w_h, w_dz, w_post, w_dA16, w_dLr16, w_hAm, w_hLm, w_z8, w_wo8,
      w_wodq, w_nscale, w_dbO, w_len, w_total;
};

// Header words at saved + s_status.
struct SavedHeader {
  int32_t status;       // device status word
  int32_t total_tiles;  // number of tiles of the actual lengths
  int32_t pad[62];
};

// Device-visible views of `saved` (fp32 arrays [B,T,U1]).
struct SavedView {
  int32_t* status;
  int32_t* total_tiles;
  int32_t* prefix;  // [B+1]
  int4* tiles;      // [max tiles]: (b, t0, u0, T_b | U_b << 16) of every actual tile
  float* lnP;       // [B]
  float *lpb, *lpl, *lnPD, *alpha, *beta;
};

struct Shape {
  int B, T, U1, H, V, blank;
};

// Position of a tile in the lattice.
struct TileCoord {
  int b, t0, u0, Tb, Ub;
};

// Binary search of the sample that owns global tile g (prefix is exclusive,
// prefix[B] = total).  Precondition: 0 <= g < prefix[B].
__device__ inline int tile_sample(const int32_t* __restrict__ prefix, int B, long long g) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((long long)__ldg(prefix + mid) <= g) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ inline TileCoord decode_tile(const int32_t* __restrict__ prefix,
                                        const int32_t* __restrict__ T_len,
                                        const int32_t* __restrict__ U_len, int B, long long g) {
  TileCoord c;
  c.b = tile_sample(prefix, B, g);
  c.Tb = __ldg(T_len + c.b);
  c.Ub = __ldg(U_len + c.b);
  long long local = g - __ldg(prefix + c.b);
  int ntu = (int)cdiv(c.Ub + 1, TU);
  c.t0 = (int)(local / ntu) * TT;
  c.u0 = (int)(local % ntu) * TU;
  return c;
}

// logaddexp with logaddexp(-inf,-inf) = -inf (never NaN).
__device__ inline float logaddexp_f(float a, float b) {
  float m = fmaxf(a, b);
  if (m == -INFINITY) return -INFINITY;
  return m + log1pf(expf(-fabsf(a - b)));
}

template <typename T> __device__ inline float to_f(T x);
template <> __device__ inline float to_f<float>(float x) { return x; }
template <> __device__ inline float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

}  // namespace rnnt
