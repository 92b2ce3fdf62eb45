// k_simt.cu -- fp32 FFMA kernels of the RNN-T joint/output/loss path.
//
// This is the path of RNNT_F32 problems: every product and sum in fp32 on the
// CUDA cores (fp32 tensor-core modes round operands to tf32, which cannot meet
// fp32 tolerances).  The steps are those of the sample-wise transducer paper
// ("Neural transducer training: reduced memory consumption with sample-wise
// computation", §2): joint network (Eq. 3-4), output layer (Eq. 5-6), the
// softmax denominator and the two log-probabilities the loss needs (Eq. 7),
// and, in the backward, dh (Eq. 10) followed by the output-layer and joint
// backward (§4).  Per chunk of tiles the scores live in the chunk buffer only
// (the Flash RNN-T blog's tiling); the chunk's z and scores are recomputed in
// the backward and the scores are overwritten with their gradients.
#include "kernels.h"

namespace rnnt {

// ---------------------------------------------------------------------------
// Generic fp32 GEMM with arbitrary strides: 64x64 output tile, k-step 16,
// 256 threads x (4x4) outputs.
constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16;

__device__ inline float ld_any(const void* p, long long i, int is_bf16) {
  return is_bf16 ? __bfloat162float(((const __nv_bfloat16*)p)[i]) : ((const float*)p)[i];
}

__device__ inline bool k_ok(const SimtGemm& g, int k) {
  if (k >= g.K) return false;
  if (!g.kmask_len) return true;
  const int q = k / g.kperiod, r = k - q * g.kperiod;
  return r < __ldg(g.kmask_len + q) + g.kmask_off;
}

__global__ void __launch_bounds__(256) k_simt_gemm(SimtGemm g) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Bs[SG_BK][SG_BN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const long long m0 = (long long)blockIdx.y * SG_BM;
  const int n0 = blockIdx.x * SG_BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += SG_BK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + 256 * i;
      {  // A tile: 64 (m) x 16 (k)
        const int mm = e >> 4, kk = e & 15;
        const long long m = m0 + mm;
        const int k = k0 + kk;
        float v = 0.f;
        if (m < g.M && k_ok(g, k)) v = ld_any(g.A, m * g.sam + (long long)k * g.sak, g.a_bf16);
        As[kk][mm] = v;
      }
      {  // B tile: 16 (k) x 64 (n)
        const int kk = e >> 6, nn = e & 63;
        const int k = k0 + kk, n = n0 + nn;
        float v = 0.f;
        if (n < g.N && k_ok(g, k))
          v = ld_any(g.Bm, (long long)k * g.sbk + (long long)n * g.sbn, g.b_bf16);
        Bs[kk][nn] = v;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long m = m0 + ty * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= g.N) continue;
      float v = g.alpha * acc[i][j];
      if (g.bias) v += ld_any(g.bias, n, g.bias_bf16);
      float* c = g.C + m * g.ldc + n;
      if (g.accumulate) v += *c;
      *c = v;
    }
  }
}

cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  if (cdiv(g.M, SG_BM) > 65535) return cudaErrorInvalidValue;
  dim3 grid((unsigned)cdiv(g.N, SG_BN), (unsigned)cdiv(g.M, SG_BM));
  k_simt_gemm<<<grid, 256, 0, s>>>(g);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Per-tile helpers.  One block per tile of the chunk; the tile's coordinates
// are decoded once into shared memory.
struct TileInfo {
  int exists, b, t0, u0, Tb, Ub;
};

__device__ inline void load_tile_info(const ChunkArgs& c, long long tile_local, TileInfo* ti) {
  if (threadIdx.x == 0) {
    const long long g = c.first_tile + tile_local;
    const int total = *c.sv.total_tiles;
    TileInfo x{};
    if (g < total) {
      TileCoord tc = decode_tile(c.sv.prefix, c.T_len, c.U_len, c.sh.B, g);
      x.exists = 1; x.b = tc.b; x.t0 = tc.t0; x.u0 = tc.u0; x.Tb = tc.Tb; x.Ub = tc.Ub;
    }
    *ti = x;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(256)
k_build_z(ChunkArgs c, const float* __restrict__ pA, const float* __restrict__ pL, void* Z,
          int z_bf16) {
  __shared__ TileInfo ti;
  load_tile_info(c, blockIdx.x, &ti);
  const int H = c.sh.H;
  const long long row0 = (long long)blockIdx.x * TILE;
  for (int e = threadIdx.x; e < TILE * H; e += blockDim.x) {
    const int i = e / H, k = e - i * H;
    const int t = ti.t0 + i / TU, u = ti.u0 + i % TU;
    float z = 0.f;
    if (ti.exists && t < ti.Tb && u <= ti.Ub) {
      z = tanhf(pA[((size_t)ti.b * c.sh.T + t) * H + k] + pL[((size_t)ti.b * c.sh.U1 + u) * H + k]);
    }
    const long long r = row0 + i;
    if (z_bf16) ((__nv_bfloat16*)Z)[r * H + k] = __float2bfloat16_rn(z);
    else ((float*)Z)[r * H + k] = z;
  }
}

cudaError_t launch_build_z(const ChunkArgs& c, const float* pA, const float* pL, void* Z,
                           int z_bf16, cudaStream_t s) {
  if (c.ntiles <= 0) return cudaSuccess;
  k_build_z<<<(unsigned)c.ntiles, 256, 0, s>>>(c, pA, pL, Z, z_bf16);
  return cudaGetLastError();
}

// One warp per lattice position (row of the chunk).
__device__ inline bool row_cell(const ChunkArgs& c, const TileInfo& ti, int i, int* t, int* u) {
  *t = ti.t0 + i / TU;
  *u = ti.u0 + i % TU;
  return ti.exists && *t < ti.Tb && *u <= ti.Ub;
}

__device__ inline float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ inline float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(256) k_lse_rows(ChunkArgs c, const float* __restrict__ Hs) {
  __shared__ TileInfo ti;
  load_tile_info(c, blockIdx.x, &ti);
  const int V = c.sh.V, lane = threadIdx.x & 31;
  for (int i = threadIdx.x >> 5; i < TILE; i += blockDim.x >> 5) {
    int t, u;
    if (!row_cell(c, ti, i, &t, &u)) continue;
    const float* h = Hs + ((long long)blockIdx.x * TILE + i) * V;
    float m = -INFINITY;
    for (int v = lane; v < V; v += 32) m = fmaxf(m, h[v]);
    m = warp_max(m);
    float sum = 0.f;
    for (int v = lane; v < V; v += 32) sum += expf(h[v] - m);
    sum = warp_sum(sum);
    if (lane == 0) {
      const float lnPD = m + logf(sum);
      const size_t cell = ((size_t)ti.b * c.sh.T + t) * c.sh.U1 + u;
      c.sv.lnPD[cell] = lnPD;
      c.sv.lpb[cell] = h[c.sh.blank] - lnPD;
      c.sv.lpl[cell] =
          (u < ti.Ub) ? h[c.labels[(size_t)ti.b * c.sh.U1 + u + 1]] - lnPD : -INFINITY;
    }
  }
}

cudaError_t launch_lse_rows(const ChunkArgs& c, const float* Hs, cudaStream_t s) {
  if (c.ntiles <= 0) return cudaSuccess;
  k_lse_rows<<<(unsigned)c.ntiles, 256, 0, s>>>(c, Hs);
  return cudaGetLastError();
}

// dh_v = g_b ((pb + pl) softmax_v - pb [v = blank] - pl [v = label]) with the
// posteriors pb = exp(alpha + lpb + beta(t+1,u) - lnP), pl = exp(alpha + lpl +
// beta(t,u+1) - lnP); beta(T_b,U_b) := 0, beta(T_b,u<U_b) := -inf.
__global__ void __launch_bounds__(256)
k_dh_rows(ChunkArgs c, float* __restrict__ Hs, const float* __restrict__ grad_loss) {
  __shared__ TileInfo ti;
  load_tile_info(c, blockIdx.x, &ti);
  const int V = c.sh.V, lane = threadIdx.x & 31, U1 = c.sh.U1;
  for (int i = threadIdx.x >> 5; i < TILE; i += blockDim.x >> 5) {
    float* h = Hs + ((long long)blockIdx.x * TILE + i) * V;
    int t, u;
    if (!row_cell(c, ti, i, &t, &u)) {
      for (int v = lane; v < V; v += 32) h[v] = 0.f;
      continue;
    }
    const size_t cell = ((size_t)ti.b * c.sh.T + t) * U1 + u;
    const float lnP = c.sv.lnP[ti.b];
    const float a = c.sv.alpha[cell];
    float bn;
    if (t + 1 < ti.Tb) bn = c.sv.beta[cell + U1];
    else bn = (u == ti.Ub) ? 0.f : -INFINITY;
    const float pb = expf(a + c.sv.lpb[cell] + bn - lnP);
    const float pl = (u < ti.Ub) ? expf(a + c.sv.lpl[cell] + c.sv.beta[cell + 1] - lnP) : 0.f;
    const int y = (u < ti.Ub) ? c.labels[(size_t)ti.b * U1 + u + 1] : -1;
    const float g = grad_loss ? grad_loss[ti.b] : 1.f;
    const float lnPD = c.sv.lnPD[cell];
    const float gam = pb + pl;
    for (int v = lane; v < V; v += 32) {
      float d = gam * expf(h[v] - lnPD);
      if (v == c.sh.blank) d -= pb;
      if (v == y) d -= pl;
      h[v] = g * d;
    }
  }
}

cudaError_t launch_dh_rows(const ChunkArgs& c, float* Hs, const float* grad_loss,
                           cudaStream_t s) {
  if (c.ntiles <= 0) return cudaSuccess;
  k_dh_rows<<<(unsigned)c.ntiles, 256, 0, s>>>(c, Hs, grad_loss);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(256)
k_da_reduce(ChunkArgs c, const float* __restrict__ dZ, const void* __restrict__ Z, int z_bf16,
            float* __restrict__ dA, float* __restrict__ dLr) {
  __shared__ TileInfo ti;
  load_tile_info(c, blockIdx.x, &ti);
  if (!ti.exists) return;
  const int H = c.sh.H;
  const long long row0 = (long long)blockIdx.x * TILE;
  for (int e = threadIdx.x; e < TILE * H; e += blockDim.x) {
    const int i = e / H, k = e - i * H;
    int t, u;
    if (!row_cell(c, ti, i, &t, &u)) continue;
    const long long r = row0 + i;
    const float z = z_bf16 ? __bfloat162float(((const __nv_bfloat16*)Z)[r * H + k])
                           : ((const float*)Z)[r * H + k];
    const float da = dZ[r * H + k] * (1.f - z * z);
    atomicAdd(dA + ((size_t)ti.b * c.sh.T + t) * H + k, da);
    atomicAdd(dLr + ((size_t)ti.b * c.sh.U1 + u) * H + k, da);
  }
}

cudaError_t launch_da_reduce(const ChunkArgs& c, const float* dZ, const void* Z, int z_bf16,
                             float* dA, float* dLr, cudaStream_t s) {
  if (c.ntiles <= 0) return cudaSuccess;
  k_da_reduce<<<(unsigned)c.ntiles, 256, 0, s>>>(c, dZ, Z, z_bf16, dA, dLr);
  return cudaGetLastError();
}

// Column sums: block (x = column strip of 256, y = row slab), atomics at the end.
__global__ void __launch_bounds__(256)
k_colsum(const float* __restrict__ X, long long R, int N, long long ld, float* __restrict__ out,
         long long rows_per) {
  const int n = blockIdx.x * 256 + threadIdx.x;
  if (n >= N) return;
  const long long r0 = (long long)blockIdx.y * rows_per;
  const long long r1 = min(R, r0 + rows_per);
  float s = 0.f;
  for (long long r = r0; r < r1; ++r) s += X[r * ld + n];
  atomicAdd(out + n, s);
}

cudaError_t launch_colsum(const float* X, long long R, int N, long long ld, float* out,
                          cudaStream_t s) {
  if (R <= 0 || N <= 0) return cudaSuccess;
  long long rows_per = 256;
  if (cdiv(R, rows_per) > 65535) rows_per = cdiv(R, 65535);
  dim3 grid((unsigned)cdiv(N, 256), (unsigned)cdiv(R, rows_per));
  k_colsum<<<grid, 256, 0, s>>>(X, R, N, ld, out, rows_per);
  return cudaGetLastError();
}

}  // namespace rnnt
