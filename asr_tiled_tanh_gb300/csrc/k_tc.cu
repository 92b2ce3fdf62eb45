// k_tc.cu -- bf16 tensor-core path of the RNN-T joint/output/loss library.
//
// One warp-specialized, persistent tcgen05 GEMM kernel serves every dense
// contraction of the path; what differs is the epilogue that consumes each
// 128 x BN fp32 accumulator tile from TMEM:
//   EPI_STORE  C = A B^T (+ bias)           joint projections, dh^A, dh^L
//   EPI_ATOMIC C += A B (split-K, fp32 red)  dW^O, dW^A, dW^L
//   EPI_LSE    scores -> online log-sum-exp over V, blank/label log-probs
//              (f^W_1 of Eq. 7 plus the gather of the two probabilities the
//              Flash RNN-T kernel emits instead of a softmax)
//   EPI_LSEK   EPI_LSE that also writes the scores (bf16, TMA stores) for
//              the untiled mode, which keeps them instead of recomputing
//   EPI_DH     scores -> dh = dL/dh (Eq. 10), written into the tile buffer
//              that holds the scores in the untiled mode (Flash RNN-T blog,
//              "Compute it, use it, make room": gradients replace scores)
//   EPI_DA     dz -> da = dz (1 - z^2), reduced over u into dA[b,t] and over
//              t into dLr[b,u] (joint-network backward, sample-wise paper §4)
// Rows of the lattice GEMMs are lattice positions: M tile m of a chunk is the
// TT x TU lattice tile (chunk's first tile + m), one position per TMEM lane.
//
// Roles: warp 0 issues TMA loads into a ring of shared-memory stages, warp 1
// allocates TMEM and one thread issues tcgen05.mma into one of two TMEM
// accumulators, and 8, 12 or 16 epilogue warps (by epilogue) drain the other
// accumulator (tcgen05.ld).  mbarriers link the roles; every wait is bounded
// and a timeout sets RNNT_ERR_TIMEOUT in the status word and winds the CTA
// down.  Kernels launch as programmatic dependents of the stream's previous
// kernel (set-up overlaps its tail; griddepcontrol.wait before any read).
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "kernels.h"
#include "profile.h"
#include "streams.h"
#include "ptx.cuh"
#include "tc.h"
#include "../../include/rnnt_testing.h"

namespace rnnt {

namespace {

constexpr int BM = 128;              // rows per tile (TMEM lanes)
constexpr int BK = 64;               // K per stage: one 128-byte swizzle atom of bf16
constexpr int EPI_WARP0 = 2;         // first epilogue warp
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s per wait, then give up
constexpr int SMEM_LIMIT = 232448;   // 227 KiB opt-in maximum per block

enum { EPI_STORE = 0, EPI_ATOMIC = 1, EPI_LSE = 2, EPI_DH = 3, EPI_DA = 4, EPI_LSEK = 5 };
constexpr bool lse_like(int e) { return e == EPI_LSE || e == EPI_LSEK; }
// epilogues that write 32 x 32 bf16 boxes through a per-warp staging area
constexpr bool box_store(int e) { return e == EPI_DH || e == EPI_LSEK; }
enum { TILES_NONE = 0, TILES_ON_M = 1, TILES_ON_K = 2 };

// Per-epilogue-warp shared scratch: either 32 rows x 16 fp32 (+1 pad) for
// column transposes, or 32 rows x 32 bf16 at an 80-byte pitch for staging
// row chunks so that global accesses cover 8 rows x 64 B per instruction.
constexpr int WSCR_BYTES = 2560;
constexpr int STAGE_PITCH = 80;

struct TcParams {
  int M, N, K;
  int m_tiles, n_tiles, k_splits, kb_total, kb_per_split;
  int units;
  int row_complete;      // a unit is one M tile with all of its N tiles, in order
  int n_split;           // row-complete units: N tiles split into this many units (1 for LSE)
  int n_split_auto;      // n_split is a maximum: the kernel picks the split from the
                         // batch's tile count (whole waves of row units)
  float* C;              // STORE / ATOMIC output, row-major with ldc
  __nv_bfloat16* Cb;     // STORE: bf16 output instead of C (row-major with ldc)
  long long ldc;
  const __nv_bfloat16* bias;  // STORE / LSE / DH: bias along N (may be NULL)
  int sbias;             // LSE / DH: the bias is copied to shared memory (N % 8 == 0)
  ChunkArgs ch;          // lattice epilogues: chunk, lengths, labels, saved arrays
  const float* grad_loss;
  const float* nscale;   // e4m3 score GEMMs: dequantization scale per N tile (NULL: 1)
  __nv_bfloat16* Hout;   // LSE: kept scores (untiled) [rows][N]; DH: dh [rows][N]
  const __nv_bfloat16* Zin;  // DA: z [rows][N]
  float* dA;
  float* dLr;
  float* dbO;            // DH: column sums of dh accumulated here (may be NULL)
  const float4* post;    // DH: per-row records (see k_posteriors)
  int32_t* status;
  // Lattice GEMMs: which axis runs over the chunk's tiles (TILES_ON_M: M
  // tiles are lattice tiles; TILES_ON_K: K runs over the tiles' rows), so
  // that units past the batch's last tile (the host sizes the chunk by an
  // upper bound) are skipped; TILES_NONE for the other GEMMs.
  int tiles_on;
  unsigned long long wait_ns;  // limit of every mbarrier wait (0: WAIT_NS)
  int skip_first_fill;         // test hook: the producer never fills the first stage
};

// Epilogue warps of a kernel, four per TMEM lane quarter for the scores
// (LSE) epilogue and three for the dh and kept-score epilogues, whose
// per-element work would otherwise hold the MMAs back (these need the 128
// registers a thread gets in a 448-thread block; LSE fits the 96 of a
// 576-thread one); two per quarter for the others.
template <int EPI>
constexpr int epi_warps() {
  return EPI == EPI_LSE ? 16 : (box_store(EPI) ? 12 : 8);
}

template <int BN, int EPI>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int EW = epi_warps<EPI>();
  static constexpr int PARTS = EW / 4;                   // warps per TMEM lane quarter
  static constexpr int THREADS = 64 + 32 * EW;
  // per epilogue warp staging area: none for LSE, a 32 x 64 B TMA-store box
  // for dh and kept scores, transposes / row staging for the others
  static constexpr int WSCR = EPI == EPI_LSE ? 0 : (box_store(EPI) ? 2048 : WSCR_BYTES);
  static constexpr int EPI_SCRATCH = EW * WSCR;
  // LSE: partials of the other parts of each row, double-buffered
  static constexpr int COMB_BYTES = lse_like(EPI) ? 2 * (PARTS - 1) * 128 * 4 * 4 : 0;
  static constexpr int BAR_BYTES = 256;
  static constexpr int STAGES_RAW =
      (SMEM_LIMIT - 1024 - EPI_SCRATCH - COMB_BYTES - BAR_BYTES) / STAGE;
  static constexpr int STAGES = STAGES_RAW > 6 ? 6 : STAGES_RAW;
  static constexpr int SMEM = 1024 + STAGES * STAGE + EPI_SCRATCH + COMB_BYTES + BAR_BYTES;
  static constexpr int TMEM_COLS = 2 * BN <= 32 ? 32 : (2 * BN <= 64 ? 64 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512)));
};

struct Unit {
  int m, n0, n1, kb0, kb1;  // M tile, N tiles [n0,n1), K blocks [kb0,kb1)
};

// Unit u of a GEMM.  Row-complete units: M tile, then the V split of its N
// tiles.  Other units: N fastest, then M, then the K split, so that the CTAs
// working at the same time share K ranges and each K block of A and B is
// fetched from DRAM about once and served to the other units from L2.
__device__ __forceinline__ Unit unit_of(const TcParams& p, int u, int kb_lim, int kbps, int ns) {
  Unit w;
  int rest = u;
  if (p.row_complete) {
    const int per = (p.n_tiles + ns - 1) / ns;
    const int sp = rest % ns;
    w.m = rest / ns;
    w.n0 = sp * per; w.n1 = min(p.n_tiles, w.n0 + per);
    w.kb0 = 0; w.kb1 = (w.n1 > w.n0) ? p.kb_total : 0;
  } else {
    const int n = rest % p.n_tiles;
    rest /= p.n_tiles;
    const int mt = rest % p.m_tiles;
    const int ks = rest / p.m_tiles;
    w.m = mt;
    w.n0 = n; w.n1 = n + 1;
    w.kb0 = ks * kbps;
    w.kb1 = min(kb_lim, w.kb0 + kbps);
  }
  return w;
}

__device__ __forceinline__ void report_timeout(const TcParams& p, volatile int* abort_flag) {
  *abort_flag = 1;
  if (p.status) atomicOr(p.status, status_bit(RNNT_ERR_TIMEOUT));
}

// Lattice coordinates of M tile m of a chunk, and of one of its rows (TMEM lane).
struct TileRef {
  bool exists;  // the tile is one of the actual tiles of the batch
  int b, t0, u0, Tb, Ub;
};

__device__ __forceinline__ TileRef tile_ref(const ChunkArgs& c, int m) {
  TileRef r{};
  const long long g = c.first_tile + m;
  if (m >= c.ntiles || g >= *c.sv.total_tiles) return r;
  const int4 e = __ldg(c.sv.tiles + g);  // (b, t0, u0, T_b | U_b << 16)
  r.exists = true;
  r.b = e.x; r.t0 = e.y; r.u0 = e.z; r.Tb = e.w & 0xffff; r.Ub = e.w >> 16;
  return r;
}

struct RowCell {
  bool valid;   // inside its sample's lattice
  int b, t, u, Tb, Ub;
};

// Whether tile m of a chunk is read by any GEMM: the actual tiles only (the
// chunk itself is sized by an upper bound, and the GEMMs skip the rest).
__device__ __forceinline__ bool tile_in_use(const ChunkArgs& c, int m) {
  return (long long)m < (long long)*c.sv.total_tiles - c.first_tile;
}

__device__ __forceinline__ RowCell row_of(const TileRef& tr, int row) {
  RowCell r{};
  r.b = tr.b; r.Tb = tr.Tb; r.Ub = tr.Ub;
  r.t = tr.t0 + row / TU;
  r.u = tr.u0 + row % TU;
  r.valid = tr.exists && r.t < tr.Tb && r.u <= tr.Ub;
  return r;
}

__device__ __forceinline__ float bf(const __nv_bfloat16* p, long long i) {
  return __bfloat162float(p[i]);
}

// 32 bias values of columns col0.. as packed bf16 (0 beyond N or without a
// bias); widened with unpack32 where they are used.  sb: the CTA's copy of the
// bias in shared memory (all lanes read the same 16 bytes: broadcasts), or NULL.
__device__ __forceinline__ void load_bias_q(const __nv_bfloat16* bias, int N, int col0,
                                            uint4 (&q)[4], const uint4* sb = nullptr) {
  if (sb && col0 + 32 <= N) {
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = sb[col0 / 8 + i];
    return;
  }
  if (bias && col0 + 32 <= N && (N & 7) == 0) {
    const uint4* src = (const uint4*)(bias + col0);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = __ldg(src + i);
    return;
  }
  const unsigned short* b16 = (const unsigned short*)bias;
  uint32_t w[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int c = col0 + 2 * k;
    const uint32_t lo = (bias && c < N) ? b16[c] : 0u;
    const uint32_t hi = (bias && c + 1 < N) ? b16[c + 1] : 0u;
    w[k] = lo | (hi << 16);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// 32 bf16 values (four 16-byte words) widened to fp32.
__device__ __forceinline__ void unpack32(const uint4 (&q)[4], float (&out)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[i * 8 + 0] = ptx::bf16lo(q[i].x); out[i * 8 + 1] = ptx::bf16hi(q[i].x);
    out[i * 8 + 2] = ptx::bf16lo(q[i].y); out[i * 8 + 3] = ptx::bf16hi(q[i].y);
    out[i * 8 + 4] = ptx::bf16lo(q[i].z); out[i * 8 + 5] = ptx::bf16hi(q[i].z);
    out[i * 8 + 6] = ptx::bf16lo(q[i].w); out[i * 8 + 7] = ptx::bf16hi(q[i].w);
  }
}

// The warp's 32 rows x 32 bf16 (columns col0 ..) of a row-major matrix, for
// lane = row: issue_rows_bf16 starts coalesced loads (8 rows x 64 B per
// instruction) early; finish_rows_bf16 redistributes them through the warp's
// staging area (80-byte pitch) when the values are needed.
__device__ __forceinline__ void issue_rows_bf16(const __nv_bfloat16* gbase, long long ld,
                                                uint4 (&x)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2), piece = lane & 3;
    x[i] = __ldg((const uint4*)(gbase + (long long)r * ld + piece * 8));
  }
}
__device__ __forceinline__ void finish_rows_bf16(unsigned char* stg, const uint4 (&x)[4],
                                                 uint4 (&q)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2), piece = lane & 3;
    *(uint4*)(stg + r * STAGE_PITCH + piece * 16) = x[i];
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = *(const uint4*)(stg + lane * STAGE_PITCH + i * 16);
  __syncwarp();
}

__device__ __forceinline__ uint4 pack8_bf16(const float* d) {
  return make_uint4(ptx::pack_bf16x2(d[0], d[1]), ptx::pack_bf16x2(d[2], d[3]),
                    ptx::pack_bf16x2(d[4], d[5]), ptx::pack_bf16x2(d[6], d[7]));
}

// Select v[j] for a runtime j in [0,32) without local memory.
__device__ __forceinline__ float pick32(const float* v, int j) {
  float r = 0.f;
#pragma unroll
  for (int k = 0; k < 32; ++k) r = (k == j) ? v[k] : r;
  return r;
}

// ---- lattice epilogues, per TMEM lane (one lattice position per thread) ----
constexpr float kLog2e = 1.4426950408889634f;

// f^W_1 (Eq. 7) as an online log-sum-exp over the V scores of the position,
// plus the blank and label scores; only these leave the SM.
struct LseState {
  float run_max, run_sum, h_blank, h_lab;
  int lab;
};

__device__ __forceinline__ void lse_init(LseState& st, const TcParams& p, const RowCell& rc) {
  st.run_max = -INFINITY;
  st.run_sum = 0.f;
  st.h_blank = 0.f;
  st.h_lab = 0.f;
  st.lab = (rc.valid && rc.u < rc.Ub) ? p.ch.labels[(size_t)rc.b * p.ch.sh.U1 + rc.u + 1] : -1;
}

// 32 scores v[] (accumulator values, bias not yet added) of columns col0.. .
// sc: the accumulator's dequantization scale (1 for bf16 operands; the same
// instruction count as a plain add).  On return v holds the scores (columns
// past V: -inf) of a lattice row.
__device__ __forceinline__ void lse_chunk(LseState& st, const TcParams& p, const RowCell& rc,
                                          float* v, const float* bb, int col0, float sc) {
  // (rows outside every lattice run through too, on their zero z rows: no
  // divergent branch; lse_finish writes nothing for them)
  const int nv = min(32, p.N - col0);
  const float2 s2 = make_float2(sc, sc);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float2 x = __ffma2_rn(make_float2(v[j], v[j + 1]), s2, make_float2(bb[j], bb[j + 1]));
    v[j] = x.x;
    v[j + 1] = x.y;
  }
  if (nv < 32) {  // columns past V take no part in the sum
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = (j < nv) ? v[j] : -INFINITY;
  }
  float cm = fmaxf(v[0], v[1]);
#pragma unroll
  for (int j = 2; j < 32; j += 2) cm = ptx::max3(cm, v[j], v[j + 1]);
  const float nm = fmaxf(st.run_max, cm);
  float s = st.run_sum * ptx::ex2((st.run_max - nm) * kLog2e);
  const float nmL = nm * kLog2e;
  const float2 l2 = make_float2(kLog2e, kLog2e), m2 = make_float2(-nmL, -nmL);
  float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const float2 y0 = __ffma2_rn(make_float2(v[j], v[j + 1]), l2, m2);
    const float2 y1 = __ffma2_rn(make_float2(v[j + 2], v[j + 3]), l2, m2);
    a0 = __fadd2_rn(a0, make_float2(ptx::ex2(y0.x), ptx::ex2(y0.y)));
    a1 = __fadd2_rn(a1, make_float2(ptx::ex2(y1.x), ptx::ex2(y1.y)));
  }
  a0 = __fadd2_rn(a0, a1);
  s += a0.x + a0.y;
  st.run_sum = s;
  st.run_max = nm;
  const int jb = p.ch.sh.blank - col0;
  if (jb >= 0 && jb < 32) st.h_blank = pick32(v, jb);
  const int jl = st.lab - col0;
  if (jl >= 0 && jl < 32) st.h_lab = pick32(v, jl);
}

__device__ __forceinline__ void lse_finish(const LseState& st, const TcParams& p,
                                           const RowCell& rc) {
  if (!rc.valid) return;
  const SavedView& sv = p.ch.sv;
  const size_t cell = ((size_t)rc.b * p.ch.sh.T + rc.t) * p.ch.sh.U1 + rc.u;
  const float ld = st.run_max + __logf(st.run_sum);
  sv.lnPD[cell] = ld;
  sv.lpb[cell] = st.h_blank - ld;
  sv.lpl[cell] = (rc.u < rc.Ub) ? st.h_lab - ld : -INFINITY;
}

// f^W_4 (Eq. 10): dh_v = g ((pb + pl) softmax_v - pb [v = blank] - pl [v = label]).
// Every column but the blank and the label one is g (pb + pl) softmax_v; those
// two come finished in the row's record and overwrite their column.
struct DhState {
  float lgn;       // log2|g (pb + pl)| - lnPD log2(e): |g (pb+pl)| softmax_v = 2^(h_v log2 e + lgn)
  float dhb, dhl;  // dh of the blank column and of the label column
  bool neg;        // g (pb + pl) < 0 (the incoming gradient of the row's sample is negative)
  int lab;         // label id of the row's label transition, -1 without one
};

// The row's record, precomputed by k_posteriors (see there for the formulas).
__device__ __forceinline__ DhState dh_state(const float4 q) {
  DhState st;
  st.lgn = q.x;
  st.dhb = q.y;
  st.dhl = q.z;
  const uint32_t w = __float_as_uint(q.w);
  st.lab = (int)(w & 0x7fffffffu) - 1;
  st.neg = (w >> 31) != 0;
  return st;
}

// Record of a row outside every lattice: dh = 0 everywhere.
__device__ __forceinline__ float4 dh_record_none() {
  return make_float4(-INFINITY, 0.f, 0.f, __uint_as_float(0u));
}

// A warp's 32 x 32 block d (lane = row) as bf16 into rows wrow0 .. +31,
// columns col0 .. +31 of the map's matrix, by a TMA store from the warp's
// staging area (32 rows x 64 bytes, 64-byte swizzle: lane r writes its
// 16-byte piece j at piece j ^ ((r >> 1) & 3), which spreads every 8 lanes
// over all 32 banks).  The store engine clips rows and columns past the
// matrix.  All lanes take part; the staging area is reused only after the
// previous store from it has been read out.
// fb / fl: this lane's row replaces column jb / jl of the block with vb / vl
// (at most two columns per row; same column: same value).
__device__ __forceinline__ void store_box_bf16(const float (&d)[32], unsigned char* stg,
                                               const CUtensorMap* tmC, int col0,
                                               long long wrow0, bool fb = false, int jb = 0,
                                               float vb = 0.f, bool fl = false, int jl = 0,
                                               float vl = 0.f) {
  const int lane = threadIdx.x & 31;
  uint4 q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = pack8_bf16(d + 8 * i);
  if (lane == 0) ptx::bulk_wait_read();
  __syncwarp();
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) *(uint4*)(stg + lane * 64 + ((i ^ sw) << 4)) = q[i];
  if (fb)
    *(__nv_bfloat16*)(stg + lane * 64 + (((jb >> 3) ^ sw) << 4) + (jb & 7) * 2) =
        __float2bfloat16_rn(vb);
  if (fl)
    *(__nv_bfloat16*)(stg + lane * 64 + (((jl >> 3) ^ sw) << 4) + (jl & 7) * 2) =
        __float2bfloat16_rn(vl);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ptx::tma_store_2d(tmC, stg, col0, (int)wrow0);
    ptx::bulk_commit();
  }
}

// dh of 32 columns (Eq. 10: softmax times the position's occupancy minus the
// blank / label posteriors).  The warp's 32 rows are written as bf16 to rows
// wrow0 .. +31 of the dh buffer (store_box_bf16); rows outside the lattice
// are 0.  When dbO is given, the block's column sums
// (of the bf16 values, read back from the staging area: lane k + 16 h sums
// columns 2k, 2k+1 over rows 16h .. 16h+15, rows of the two halves taken in
// opposite parity so that the reads hit distinct banks) are added to it.
// bq: the 32 bias values (packed bf16).  All lanes take part.
__device__ __forceinline__ void dh_chunk(const DhState& st, const TcParams& p, const RowCell& rc,
                                         float (&d)[32], const uint4 (&bq)[4], int col0,
                                         long long wrow0, unsigned char* stg,
                                         const CUtensorMap* tmC, bool write, float sc) {
  // d holds the chunk's scores on entry and dh on exit.  Rows outside every
  // lattice need no branch: their z rows are 0 and their record's lgn is
  // -inf, so every column comes out 0 (and their blank/label values are 0).
  const int nv = min(32, p.N - col0);
  {
    // g (pb + pl) softmax_v for every column; the blank and label terms are
    // applied only to the (at most two) columns they belong to
    // (pairs of columns through the packed fp32 add / fma)
    // (sc: the accumulator's dequantization scale, 1 for bf16 operands)
    const float2 l2 = make_float2(kLog2e, kLog2e), g2 = make_float2(st.lgn, st.lgn);
    const float2 s2 = make_float2(sc, sc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w[4] = {bq[i].x, bq[i].y, bq[i].z, bq[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float& d0 = d[8 * i + 2 * k];
        float& d1 = d[8 * i + 2 * k + 1];
        const float2 x = __ffma2_rn(make_float2(d0, d1), s2,
                                    make_float2(ptx::bf16lo(w[k]), ptx::bf16hi(w[k])));
        const float2 y = __ffma2_rn(x, l2, g2);
        d0 = ptx::ex2(y.x);
        d1 = ptx::ex2(y.y);
      }
    }
    // a tile is one sample: the sign is the same on every row of the warp
    // that has one (rows outside the lattice are 0 either way)
    if (__any_sync(0xffffffffu, st.neg)) {
#pragma unroll
      for (int j = 0; j < 32; ++j) d[j] = -d[j];
    }
    if (nv < 32) {
#pragma unroll
      for (int j = 0; j < 32; ++j) d[j] = (j < nv) ? d[j] : 0.f;
    }
  }
  const int lane = threadIdx.x & 31;
  if (write && col0 < p.N) {  // (no store box starts past the last column)
    // the blank and the label column of the row take their finished values
    const int jb = p.ch.sh.blank - col0, jl = st.lab - col0;
    store_box_bf16(d, stg, tmC, col0, wrow0, (unsigned)jb < 32u, jb, st.dhb,
                   st.lab >= 0 && (unsigned)jl < 32u, jl, st.dhl);
    if (p.dbO) {
      // row 16h + 2q + (e ^ h): its 16-byte piece k/4 sits at (k/4 ^ (q & 3))
      const int k = lane & 15, h = lane >> 4;
      const uint32_t a0 = ptx::smem_u32(stg) + 1024 * h + (k & 3) * 4;
      uint32_t ad[2][4];
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int q = 0; q < 4; ++q) ad[e][q] = a0 + 64 * (e ^ h) + (((k >> 2) ^ q) << 4);
      float2 acc = make_float2(0.f, 0.f);
      auto add = [&](uint32_t w) {
        acc = __fadd2_rn(acc, make_float2(ptx::bf16lo(w), ptx::bf16hi(w)));
      };
      // q = 0..7: rows 2q, 2q+1 of the half; q & 3 selects the address, q / 4 the offset
      add(ptx::lds32<0>(ad[0][0]));   add(ptx::lds32<0>(ad[1][0]));
      add(ptx::lds32<128>(ad[0][1])); add(ptx::lds32<128>(ad[1][1]));
      add(ptx::lds32<256>(ad[0][2])); add(ptx::lds32<256>(ad[1][2]));
      add(ptx::lds32<384>(ad[0][3])); add(ptx::lds32<384>(ad[1][3]));
      add(ptx::lds32<512>(ad[0][0])); add(ptx::lds32<512>(ad[1][0]));
      add(ptx::lds32<640>(ad[0][1])); add(ptx::lds32<640>(ad[1][1]));
      add(ptx::lds32<768>(ad[0][2])); add(ptx::lds32<768>(ad[1][2]));
      add(ptx::lds32<896>(ad[0][3])); add(ptx::lds32<896>(ad[1][3]));
      float s0 = acc.x, s1 = acc.y;
      s0 += __shfl_xor_sync(0xffffffffu, s0, 16);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 16);
      if (h == 0 && col0 + 2 * k < p.N) ptx::red_add_v2(p.dbO + col0 + 2 * k, s0, s1);
    }
  }
}

// F8: A and B are e4m3 (K-major only; tcgen05.mma kind::f8f6f4, 128 elements
// = 128 bytes of K per stage, 32 per instruction) and each N tile's
// accumulator is scaled by nscale[n] in the epilogue; otherwise bf16 (kind::f16,
// 64 elements of K per stage, 16 per instruction).  A stage holds the same
// bytes either way.
template <int BN, int A_MN, int B_MN, int EPI, int F8>
__global__ void __launch_bounds__(Cfg<BN, EPI>::THREADS, 1)
k_tc_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
          const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  using C = Cfg<BN, EPI>;
  static_assert(!F8 || (!A_MN && !B_MN), "e4m3 operands are K-major");
  constexpr int BKE = F8 ? 128 : BK;     // K elements per stage
  constexpr int KSTEP = F8 ? 32 : 16;    // K elements per instruction
  const int cta = blockIdx.x, n_ctas = gridDim.x;
  const uint64_t wait_ns = p.wait_ns ? p.wait_ns : WAIT_NS;
  constexpr int STAGES = C::STAGES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sA = smem;
  unsigned char* sB = smem + STAGES * C::A_BYTES;
  float* scratch = (float*)(smem + STAGES * C::STAGE);
  float* comb = (float*)(smem + STAGES * C::STAGE + C::EPI_SCRATCH);
  uint64_t* bars = (uint64_t*)(smem + STAGES * C::STAGE + C::EPI_SCRATCH + C::COMB_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint64_t* comb_bar = done_bar + 1;  // [2]: the other parts' LSE partials are in `comb`
  uint32_t* tmem_holder = (uint32_t*)(comb_bar + 2);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);
  // score epilogues: the output bias, copied once per CTA behind the barrier
  // area when the launch provided the room (p.sbias); read as broadcasts
  uint4* sbias = (uint4*)(smem + C::SMEM - 1024);

  const int warp = ptx::warp_id(), lane = ptx::lane_id();
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);  // released by the MMA commit of the stage
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&acc_full[a], 1);
      ptx::mbar_init(&acc_empty[a], 32 * C::EW);
      ptx::mbar_init(&comb_bar[a], 128 * (C::PARTS - 1 > 0 ? C::PARTS - 1 : 1));
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  if ((lse_like(EPI) || EPI == EPI_DH) && p.sbias) {
    // (the bias is a caller input that no kernel of the stream writes: it
    // may be read before the programmatic-dependency wait)
    const uint4* src = (const uint4*)p.bias;
    for (int i = threadIdx.x; i < p.N / 8; i += blockDim.x) sbias[i] = __ldg(src + i);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Launched as the programmatic dependent of the stream's previous kernel:
  // the set-up above overlapped its tail; its results are read only from here.
  ptx::griddep_wait();
  ptx::griddep_launch();
  // units that hold actual lattice tiles: a prefix of the unit order (M
  // groups, resp. K splits, are the slow index), read from the tile count
  int units = p.units, kb_lim = p.kb_total, kbps = p.kb_per_split;
  int ns = max(1, p.n_split);  // row-complete units: V split of a tile
  if (p.tiles_on != TILES_NONE) {
    const long long have = max(0LL, min(p.ch.ntiles, (long long)*p.ch.sv.total_tiles -
                                                         p.ch.first_tile));
    if (p.tiles_on == TILES_ON_M) {
      const int tiles = (int)have;
      // fewer than ~4 waves of tiles: each tile's V range is split over
      // several units so that the last wave is not mostly idle
      if (p.n_split_auto && tiles > 0)
        ns = max(1, min(ns, (int)((4LL * n_ctas + tiles - 1) / tiles)));
      // (row-complete: the V split is the fast index; otherwise N, with no K split)
      units = min(units, tiles * (p.row_complete ? ns : p.n_tiles));
    } else {
      kb_lim = (int)min((long long)p.kb_total, have * (BM / BK));
      // the host's split count (chosen for whole waves) over the K blocks
      // that exist: equal splits instead of fewer, full-length ones
      kbps = max(1, (kb_lim + p.k_splits - 1) / p.k_splits);
      const int splits = (kb_lim + kbps - 1) / kbps;
      units = min(units, splits * p.m_tiles * p.n_tiles);
    }
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (ptx::elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int issued[6] = {-1, -1, -1, -1, -1, -1};  // parity of the last fill per stage
      bool first_fill = true;
      for (int gi = cta; gi < units && !*abort_flag; gi += n_ctas) {
        const Unit w = unit_of(p, gi, kb_lim, kbps, ns);
        if (w.kb1 <= w.kb0) continue;
        for (int n = w.n0; n < w.n1 && !*abort_flag; ++n) {
          for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (!ptx::mbar_wait(&empty[stage], phase ^ 1, wait_ns)) {
              report_timeout(p, abort_flag);
              break;
            }
            if (p.skip_first_fill && first_fill) {  // test hook: leave this stage empty
              first_fill = false;
              if (++stage == STAGES) { stage = 0; phase ^= 1; }
              continue;
            }
            first_fill = false;
            ptx::mbar_arrive_expect_tx(&full[stage], C::STAGE);
            unsigned char* a = sA + stage * C::A_BYTES;
            unsigned char* b = sB + stage * C::B_BYTES;
            if (!A_MN) {
              ptx::tma_load_2d(a, &tmA, &full[stage], kb * BKE, w.m * BM);
            } else {
              ptx::tma_load_2d(a, &tmA, &full[stage], w.m * BM, kb * BK);
              ptx::tma_load_2d(a + 64 * 128, &tmA, &full[stage], w.m * BM + 64, kb * BK);
            }
            if (!B_MN) {
              ptx::tma_load_2d(b, &tmB, &full[stage], kb * BKE, n * BN);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                ptx::tma_load_2d(b + j * 64 * 128, &tmB, &full[stage], n * BN + 64 * j, kb * BK);
            }
#pragma unroll
            for (int k = 0; k < 6; ++k)
              if (k == stage) issued[k] = (int)phase;
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
          }
        }
      }
      // Wind-down: every fill this thread issued must have landed before the
      // CTA may exit (normally all of them were consumed already).
#pragma unroll
      for (int s = 0; s < 6; ++s)
        if (s < STAGES && issued[s] >= 0 &&
            !ptx::mbar_wait(&full[s], (uint32_t)issued[s], wait_ns))
          report_timeout(p, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (ptx::elect_one()) {
      constexpr uint32_t IDESC =
          F8 ? ptx::idesc_e4m3(BM, BN, A_MN, B_MN) : ptx::idesc_bf16(BM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int gi = cta; gi < units && !*abort_flag; gi += n_ctas) {
        const Unit w = unit_of(p, gi, kb_lim, kbps, ns);
        if (w.kb1 <= w.kb0) continue;
        for (int n = w.n0; n < w.n1 && !*abort_flag; ++n) {
          if (!ptx::mbar_wait(&acc_empty[acc], acc_phase ^ 1, wait_ns)) {
            report_timeout(p, abort_flag);
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          bool ok = true;
          for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (!ptx::mbar_wait(&full[stage], phase, wait_ns)) {
              report_timeout(p, abort_flag);
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t a0 = ptx::smem_u32(sA + stage * C::A_BYTES);
            const uint32_t b0 = ptx::smem_u32(sB + stage * C::B_BYTES);
            // a partial last K block (K not a multiple of the stage's K)
            // issues only the steps that hold data; the rest of the stage is
            // the TMA's zero fill
            const int ksteps = min(BKE / KSTEP, (p.K - kb * BKE + KSTEP - 1) / KSTEP);
#pragma unroll
            for (int k = 0; k < BKE / KSTEP; ++k) {
              if (k >= ksteps) break;
              // K-major: one step = 32 bytes along the swizzled row (16 bf16
              // or 32 e4m3).  MN-major: 16 K rows = two 8-row groups of 1024 bytes.
              const uint64_t ad = A_MN ? ptx::sdesc_sw128(a0 + k * 2048, 64 * 128, 1024)
                                       : ptx::sdesc_sw128(a0 + k * 32, 16, 1024);
              const uint64_t bd = B_MN ? ptx::sdesc_sw128(b0 + k * 2048, 64 * 128, 1024)
                                       : ptx::sdesc_sw128(b0 + k * 32, 16, 1024);
              const uint32_t accum = (kb > w.kb0 || k > 0) ? 1u : 0u;
              if constexpr (F8) ptx::mma_e4m3(d_tmem, ad, bd, IDESC, accum);
              else ptx::mma_bf16(d_tmem, ad, bd, IDESC, accum);
            }
            ptx::mma_commit(&empty[stage]);
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          ptx::mma_commit(&acc_full[acc]);
          if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
      }
      // all issued MMAs complete before TMEM is released
      ptx::mma_commit(done_bar);
      if (!ptx::mbar_wait(done_bar, 0, wait_ns)) report_timeout(p, abort_flag);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // EW warps: warp w drains TMEM lane quarter (w & 3) and, of each
    // accumulator's 32-column chunks, those with c % PARTS == its part.  With
    // two parts the next chunk's tcgen05.ld is in flight while the current one
    // is processed; with more, the other warps of the quarter cover it.
    constexpr int PARTS = C::PARTS;
    // double-buffered TMEM loads (not for dz: its epilogue is at the register
    // limit of a 320-thread block, and the extra 32 values spill)
    constexpr bool DB = PARTS == 2 && EPI != EPI_DA;
    const int sub = warp & 3;                    // TMEM lane quarter of this warp
    const int hf = (warp - EPI_WARP0) >> 2;      // part: chunks c % PARTS == hf
    const int row = sub * 32 + lane;             // accumulator row owned by this thread
    float* wscr = (float*)((unsigned char*)scratch + (warp - EPI_WARP0) * C::WSCR);
    constexpr int NCH = BN / 32;
    int acc = 0;
    uint32_t acc_phase = 0;
    // dh epilogue: the row's record of the next unit is loaded one unit ahead
    float4 post_next = dh_record_none();
    if (EPI == EPI_DH && cta < units) {
      const Unit w0 = unit_of(p, cta, kb_lim, kbps, ns);
      if (w0.m < p.ch.ntiles) post_next = __ldg(p.post + (long long)w0.m * BM + row);
    }
    for (int gi = cta; gi < units && !*abort_flag; gi += n_ctas) {
      const Unit w = unit_of(p, gi, kb_lim, kbps, ns);
      const float4 post_cur = post_next;
      if (EPI == EPI_DH && gi + n_ctas < units) {
        const Unit wn = unit_of(p, gi + n_ctas, kb_lim, kbps, ns);
        post_next = (wn.m < p.ch.ntiles) ? __ldg(p.post + (long long)wn.m * BM + row)
                                         : dh_record_none();
      }
      if (w.kb1 <= w.kb0) continue;
      const int uidx = gi / n_ctas;   // this CTA's unit counter
      // per-unit state of the lattice epilogues
      TileRef tr{};
      RowCell rc{};
      LseState ls;
      DhState ds;
      if (lse_like(EPI) || EPI == EPI_DH || EPI == EPI_DA) {
        tr = tile_ref(p.ch, w.m);
        rc = row_of(tr, row);
      }
      if (lse_like(EPI)) lse_init(ls, p, rc);
      if (EPI == EPI_DH) ds = dh_state(post_cur);
      bool ok = true;
      for (int n = w.n0; n < w.n1; ++n) {
        if (*abort_flag || !ptx::mbar_wait(&acc_full[acc], acc_phase, wait_ns)) {
          report_timeout(p, abort_flag);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(sub * 32) << 16);
        const float sc = (F8 && p.nscale) ? __ldg(p.nscale + n) : 1.f;
        float v[32], vn[DB ? 32 : 1];
        ptx::tmem_ld32(tbase + hf * 32, v);
        // bias values of the current chunk; the next chunk's are loaded early
        constexpr bool USE_BIAS = (EPI == EPI_STORE || lse_like(EPI) || EPI == EPI_DH);
        uint4 bq[4];
        const uint4* sb = (EPI != EPI_STORE && p.sbias) ? sbias : nullptr;
        if (USE_BIAS) load_bias_q(p.bias, p.N, n * BN + hf * 32, bq, sb);
        // dz epilogue: z rows of the current chunk, loaded one chunk ahead
        const bool z_vec = (EPI == EPI_DA) && tr.exists && (p.N & 7) == 0;
        const __nv_bfloat16* zrow = p.Zin + ((long long)w.m * BM + sub * 32) * p.N;
        uint4 zx[4];
        if (EPI == EPI_DA && z_vec && n * BN + hf * 32 + 32 <= p.N)
          issue_rows_bf16(zrow + n * BN + hf * 32, p.N, zx);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(v);
#pragma unroll 1
        for (int c = hf; c < NCH; c += PARTS) {
          const bool more = c + PARTS < NCH;
          if constexpr (DB) {
            if (more) ptx::tmem_ld32(tbase + (c + 2) * 32, vn);
          }
          const int col0 = n * BN + c * 32;
          uint4 bqn[4];
          if (DB && USE_BIAS && more) load_bias_q(p.bias, p.N, col0 + 64, bqn, sb);

          float bb[32];
          if (USE_BIAS && EPI != EPI_DH) unpack32(bq, bb);
          if constexpr (EPI == EPI_STORE || EPI == EPI_ATOMIC) {
            const long long grow = (long long)w.m * BM + row;
            if (grow < p.M && col0 < p.N) {
              float* dst = p.C + grow * p.ldc + col0;
              if (EPI == EPI_STORE && p.Cb) {  // bf16 output (nearest even)
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += bb[j];
                __nv_bfloat16* db = p.Cb + grow * p.ldc + col0;
                if (col0 + 32 <= p.N && (p.ldc & 7) == 0) {
#pragma unroll
                  for (int i = 0; i < 4; ++i) *(uint4*)(db + 8 * i) = pack8_bf16(v + 8 * i);
                } else {
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    if (col0 + j < p.N) db[j] = __float2bfloat16_rn(v[j]);
                }
              } else if constexpr (EPI == EPI_STORE) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += bb[j];
                if (col0 + 32 <= p.N && (p.ldc & 3) == 0) {
#pragma unroll
                  for (int j = 0; j < 32; j += 4)
                    *(float4*)(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                } else {
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    if (col0 + j < p.N) dst[j] = v[j];
                }
              } else if (col0 + 32 <= p.N && (p.ldc & 3) == 0) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                  ptx::red_add_v4(dst + j, v[j], v[j + 1], v[j + 2], v[j + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (col0 + j < p.N) ptx::red_add_f32(dst + j, v[j]);
              }
            }
          } else if constexpr (lse_like(EPI)) {
            lse_chunk(ls, p, rc, v, bb, col0, sc);
            if constexpr (EPI == EPI_LSEK) {
              // the scores as the untiled mode keeps them (rows outside the
              // lattice: 0)
              if (!rc.valid) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
              }
              if (w.m < p.ch.ntiles && col0 < p.N)
                store_box_bf16(v, (unsigned char*)wscr, &tmC, col0,
                               (long long)w.m * BM + sub * 32);
            }
          } else if constexpr (EPI == EPI_DH) {
            dh_chunk(ds, p, rc, v, bq, col0, (long long)w.m * BM + sub * 32,
                     (unsigned char*)wscr, &tmC, w.m < p.ch.ntiles, sc);
          } else if constexpr (EPI == EPI_DA) {
            // da = dz (1 - z^2) on the thread's own row, then 16-column halves
            // of the warp's 32 x 32 block are transposed through the warp's
            // scratch (lane = column c, row half h) and summed over the tile's
            // u (into dA[b,t]) and t (into dLr[b,u]).
            // (da is formed in place in v)
            if (z_vec && col0 + 32 <= p.N) {
              uint4 zq[4];
              finish_rows_bf16((unsigned char*)wscr, zx, zq);
              // the next chunk's z is in flight while this one is processed
              if (more && col0 + 96 <= p.N) issue_rows_bf16(zrow + col0 + 64, p.N, zx);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint32_t zw[4] = {zq[i].x, zq[i].y, zq[i].z, zq[i].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float z0 = ptx::bf16lo(zw[k]), z1 = ptx::bf16hi(zw[k]);
                  v[8 * i + 2 * k] = rc.valid ? v[8 * i + 2 * k] * (1.f - z0 * z0) : 0.f;
                  v[8 * i + 2 * k + 1] = rc.valid ? v[8 * i + 2 * k + 1] * (1.f - z1 * z1) : 0.f;
                }
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const bool ok = rc.valid && col0 + j < p.N;
                const float z = ok ? bf(p.Zin, ((long long)w.m * BM + row) * p.N + col0 + j) : 0.f;
                v[j] = ok ? v[j] * (1.f - z * z) : 0.f;
              }
            }
            const int cc = lane & 15, h = lane >> 4;
            // rows r of this warp: t = tw + r / TU, u = u0 + r % TU; a 16-row
            // half holds FQ frames of TU label positions
            constexpr int FQ = 16 / TU;
            static_assert(16 % TU == 0 && TU % 2 == 0, "tile shape");
            const int tw = tr.t0 + sub * (32 / TU);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
              for (int j = 0; j < 16; ++j) wscr[lane * 17 + j] = v[half * 16 + j];
              __syncwarp();
              // this lane: column col0 + half*16 + cc, rows h*16 .. h*16+15
              // (t = tw + FQ h .. tw + FQ h + FQ-1, u = u0 .. u0+TU-1)
              float sum_u[TU], st[FQ];
#pragma unroll
              for (int q = 0; q < FQ; ++q) {
                st[q] = 0.f;
#pragma unroll
                for (int k = 0; k < TU; ++k) {
                  const float x = wscr[(h * 16 + q * TU + k) * 17 + cc];
                  st[q] += x;
                  sum_u[k] = (q == 0) ? x : sum_u[k] + x;
                }
              }
#pragma unroll
              for (int k = 0; k < TU; ++k) sum_u[k] += __shfl_xor_sync(0xffffffffu, sum_u[k], 16);
              const int col = col0 + half * 16 + cc;
              if (col < p.N && tr.exists && tw < tr.Tb) {
#pragma unroll
                for (int q = 0; q < FQ; ++q) {
                  const int t = tw + FQ * h + q;
                  if (t < tr.Tb)
                    ptx::red_add_f32(p.dA + ((size_t)tr.b * p.ch.sh.T + t) * p.N + col, st[q]);
                }
                // the two row halves split the TU label positions: h=0 takes the first half
#pragma unroll
                for (int k = 0; k < TU / 2; ++k) {
                  const int kk = h * (TU / 2) + k;
                  const float x = h ? sum_u[TU / 2 + k] : sum_u[k];
                  if (tr.u0 + kk <= tr.Ub)
                    ptx::red_add_f32(p.dLr + ((size_t)tr.b * p.ch.sh.U1 + tr.u0 + kk) * p.N + col,
                                     x);
                }
              }
              __syncwarp();
            }
          }
          if (more) {
            if constexpr (DB) {
              ptx::tmem_ld_wait();
              ptx::reg_fence32(vn);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = vn[j];
              if (USE_BIAS) {
#pragma unroll
                for (int i = 0; i < 4; ++i) bq[i] = bqn[i];
              }
            } else {
              ptx::tmem_ld32(tbase + (c + PARTS) * 32, v);
              if (USE_BIAS) load_bias_q(p.bias, p.N, col0 + 32 * PARTS, bq, sb);
              ptx::tmem_ld_wait();
              ptx::reg_fence32(v);
            }
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&acc_empty[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      if (lse_like(EPI) && ok) {
        // combine the column parts of each row: parts 1.. hand their partial
        // (max, sum, blank score, label score) to part 0
        float* cb = comb + ((uidx & 1) * (PARTS - 1)) * 128 * 4;
        if (hf > 0) {
          float* mine = cb + ((hf - 1) * 128 + row) * 4;
          mine[0] = ls.run_max;
          mine[1] = ls.run_sum;
          mine[2] = ls.h_blank;
          mine[3] = ls.h_lab;
          ptx::mbar_arrive(&comb_bar[uidx & 1]);
        } else if (ptx::mbar_wait(&comb_bar[uidx & 1], (uint32_t)(uidx >> 1) & 1u, wait_ns)) {
          float nm = ls.run_max;
#pragma unroll
          for (int q = 1; q < PARTS; ++q) nm = fmaxf(nm, cb[((q - 1) * 128 + row) * 4]);
          float sum = 0.f;
          if (ls.run_max != -INFINITY) sum += ls.run_sum * ptx::ex2((ls.run_max - nm) * kLog2e);
#pragma unroll
          for (int q = 1; q < PARTS; ++q) {
            const float* o = cb + ((q - 1) * 128 + row) * 4;
            if (o[0] != -INFINITY) sum += o[1] * ptx::ex2((o[0] - nm) * kLog2e);
          }
          ls.run_max = nm;
          ls.run_sum = sum;
          // each score column lives in exactly one part: take it from there
          const int bpart = ((p.ch.sh.blank % BN) / 32) % PARTS;
          if (bpart != 0) ls.h_blank = cb[((bpart - 1) * 128 + row) * 4 + 2];
          if (ls.lab >= 0) {
            const int lpart = ((ls.lab % BN) / 32) % PARTS;
            if (lpart != 0) ls.h_lab = cb[((lpart - 1) * 128 + row) * 4 + 3];
          }
          lse_finish(ls, p, rc);
        } else {
          report_timeout(p, abort_flag);
        }
      }
    }
    // the box stores issued by this warp are complete before the CTA ends
    if (box_store(EPI) && lane == 0) ptx::bulk_wait_all();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
}

}  // namespace
}  // namespace rnnt

// ===========================================================================
// Elementwise helpers of the tensor-core path.
namespace rnnt {
namespace {

// z rows of a chunk in bf16: tanh(pA[b,t] + pL[b,u]) (joint network, Eq. 3-4),
// 0 on rows outside the lattice.  One block per tile; a thread owns 4
// consecutive h (a column group, strided by the block size) and writes them
// for all 128 positions of the tile: the tile's TU pL rows are loaded once into
// registers, each of its TT pA rows once per frame, and the stores of a warp
// cover 256 contiguous bytes of a z row.
//
// OUT selects the outputs: bit 0 the bf16 z rows (Z, [rows][H]), bit 1 the
// e4m3 operand of the e4m3 score GEMMs (Z8, [rows][H] bytes): e4m3(z 2^8),
// rounded to nearest even (|z| < 1, so 2^8 z stays below the e4m3 maximum
// of 448; the scale is a power of two, so the GEMM's result is scaled back
// exactly).
constexpr float kZ8Scale = 256.f;
template <int OUT>
__global__ void __launch_bounds__(256)
k_build_z_bf16(ChunkArgs c, const float* __restrict__ pA, const float* __restrict__ pL,
               __nv_bfloat16* __restrict__ Z, unsigned char* __restrict__ Z8) {
  ptx::griddep_launch();  // the GEMM that follows may start its set-up
  if (!tile_in_use(c, blockIdx.x)) return;
  const TileRef tr = tile_ref(c, blockIdx.x);
  const int H = c.sh.H, H4 = H / 4;
  const int nt = tr.exists ? min(TT, tr.Tb - tr.t0) : 0;      // frames of the tile in the lattice
  const int nu = tr.exists ? min(TU, tr.Ub + 1 - tr.u0) : 0;  // label positions
  const float* gA = pA + ((size_t)tr.b * c.sh.T + tr.t0) * H;
  const float* gL = pL + ((size_t)tr.b * c.sh.U1 + tr.u0) * H;
  using ptx::pack_bf16x2;
  using ptx::tanh_approx;
  for (int k4 = threadIdx.x; k4 < H4; k4 += blockDim.x) {
    float4 l[TU];
#pragma unroll
    for (int ui = 0; ui < TU; ++ui)
      l[ui] = ui < nu ? __ldg((const float4*)(gL + (size_t)ui * H) + k4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    __nv_bfloat16* z = Z + (long long)blockIdx.x * TILE * H + 4 * k4;
    unsigned char* z8 = Z8 + (long long)blockIdx.x * TILE * H + 4 * k4;
    // four frames per pass: their pA loads are in flight together (the kernel
    // waits on these loads; two per pass left it 30% slower at B=1024, 40 s,
    // eight gained nothing)
#pragma unroll 4
    for (int ti = 0; ti < TT; ++ti) {
      const bool t_ok = ti < nt;
      const float4 a = t_ok ? __ldg((const float4*)(gA + (size_t)ti * H) + k4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int ui = 0; ui < TU; ++ui) {
        // tanh.approx (relative error ~2^-11) is below the bf16 rounding of z
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t_ok && ui < nu)
          t = make_float4(tanh_approx(a.x + l[ui].x), tanh_approx(a.y + l[ui].y),
                          tanh_approx(a.z + l[ui].z), tanh_approx(a.w + l[ui].w));
        const long long r = (long long)(ti * TU + ui) * H;
        if (OUT & 1)
          *(uint2*)(z + r) = make_uint2(pack_bf16x2(t.x, t.y), pack_bf16x2(t.z, t.w));
        if (OUT & 2)
          *(uint32_t*)(z8 + r) =
              (uint32_t)ptx::pack_e4m3x2(t.x * kZ8Scale, t.y * kZ8Scale) |
              ((uint32_t)ptx::pack_e4m3x2(t.z * kZ8Scale, t.w * kZ8Scale) << 16);
      }
    }
  }
}

// Z (bf16) and/or Z8 (e4m3) rows of a chunk; a NULL output is not written.
cudaError_t launch_build_z_bf16(const ChunkArgs& c, const float* pA, const float* pL,
                                __nv_bfloat16* Z, unsigned char* Z8, cudaStream_t s) {
  const int threads = std::min(256, (int)cdiv(c.sh.H / 4, 32) * 32);
  if (Z && Z8)
    k_build_z_bf16<3><<<(unsigned)c.ntiles, threads, 0, s>>>(c, pA, pL, Z, Z8);
  else if (Z8)
    k_build_z_bf16<2><<<(unsigned)c.ntiles, threads, 0, s>>>(c, pA, pL, Z, Z8);
  else
    k_build_z_bf16<1><<<(unsigned)c.ntiles, threads, 0, s>>>(c, pA, pL, Z, Z8);
  return cudaGetLastError();
}

// W^O quantized for the e4m3 score GEMMs, one block of 256 rows (the score
// GEMMs' N tile) per CTA: S = 2^k, the smallest power of two with
// max|W^O[block]| / S <= 448 (1 for an all-zero block); q = e4m3(W^O / S)
// (nearest even; W^O / S is exact); the dequantized matrix W^O_q = q S, exact
// in bf16 (4 significant bits), which the backward's dz GEMM uses so that the
// forward and the backward differentiate the same output layer; and
// nscale[block] = S / 2^8, the factor that turns an accumulator of
// e4m3(2^8 z) . q back into W^O_q z.
constexpr int kWBlock = 256;
__global__ void __launch_bounds__(1024)
k_quantize_wo(const __nv_bfloat16* __restrict__ WO, unsigned char* __restrict__ Q,
              __nv_bfloat16* __restrict__ Wdq, float* __restrict__ nscale, int V, int H) {
  __shared__ float red[32];
  const int v0 = blockIdx.x * kWBlock, v1 = min(V, v0 + kWBlock);
  const long long e0 = (long long)v0 * H, e1 = (long long)v1 * H;  // elements of the block
  float amax = 0.f;
  for (long long i = e0 + 2 * (long long)threadIdx.x; i < e1; i += 2 * blockDim.x) {
    const uint32_t w = *(const uint32_t*)(WO + i);  // H even: pairs never straddle rows
    amax = fmaxf(amax, fmaxf(fabsf(ptx::bf16lo(w)), fabsf(ptx::bf16hi(w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float m = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) red[0] = m;
  }
  __syncthreads();
  amax = red[0];
  // amax = f 2^e with f in [0.5, 1); 448 = 0.875 2^9
  int e = 0;
  const float f = frexpf(amax, &e);
  const int k = amax > 0.f ? e - 9 + (f > 0.875f ? 1 : 0) : 0;
  const float S = ldexpf(1.f, k), invS = ldexpf(1.f, -k);
  if (threadIdx.x == 0) nscale[blockIdx.x] = S * (1.f / kZ8Scale);
  for (long long i = e0 + 2 * (long long)threadIdx.x; i < e1; i += 2 * blockDim.x) {
    const uint32_t w = *(const uint32_t*)(WO + i);
    const uint16_t q = ptx::pack_e4m3x2(ptx::bf16lo(w) * invS, ptx::bf16hi(w) * invS);
    *(uint16_t*)(Q + i) = q;
    const float2 d = ptx::unpack_e4m3x2(q);
    *(uint32_t*)(Wdq + i) = ptx::pack_bf16x2(d.x * S, d.y * S);
  }
}

cudaError_t launch_quantize_wo(const void* WO, void* Q, void* Wdq, float* nscale, int V, int H,
                               cudaStream_t s) {
  if (V <= 0 || H <= 0) return cudaSuccess;
  k_quantize_wo<<<(unsigned)cdiv(V, kWBlock), 1024, 0, s>>>(
      (const __nv_bfloat16*)WO, (unsigned char*)Q, (__nv_bfloat16*)Wdq, nscale, V, H);
  return cudaGetLastError();
}

// Per-row records for the dh passes (f^W_4, Eq. 10).  With the posteriors
// pb = exp(alpha + lpb + beta(t+1,u) - lnP) and pl = exp(alpha + lpl +
// beta(t,u+1) - lnP) (beta(T_b,U_b) := 0, beta(T_b,u<U_b) := -inf, pl = 0 on
// row U_b), g = grad_loss[b] and G = g (pb + pl), dh_v = G softmax_v on every
// column but two: the blank column, G exp(lpb) - g pb, and the label column,
// G exp(lpl) - g pl (both terms when the label is the blank id); softmax at
// those columns is exp(lpb), exp(lpl) from the forward.  The record of a
// lattice position is
//   (log2|G| - lnPD log2(e), dh of the blank column, dh of the label column,
//    bits: label id + 1 in bits 0-30 (0: no label transition), G < 0 in bit 31);
// rows outside the lattice get dh_record_none().  One thread per row of the chunk.
__global__ void __launch_bounds__(128)
k_posteriors(ChunkArgs c, const float* __restrict__ grad_loss, float4* __restrict__ post) {
  if (!tile_in_use(c, blockIdx.x)) return;
  const TileRef tr = tile_ref(c, blockIdx.x);
  const RowCell rc = row_of(tr, threadIdx.x);
  float4 rec = dh_record_none();
  if (rc.valid) {
    const SavedView& sv = c.sv;
    const int U1 = c.sh.U1;
    const size_t cell = ((size_t)rc.b * c.sh.T + rc.t) * U1 + rc.u;
    const float lnP = sv.lnP[rc.b];
    const float a = sv.alpha[cell];
    float bn;
    if (rc.t + 1 < rc.Tb) bn = sv.beta[cell + U1];
    else bn = (rc.u == rc.Ub) ? 0.f : -INFINITY;
    const float lpb = sv.lpb[cell];
    const bool has_lab = rc.u < rc.Ub;
    const float lpl = has_lab ? sv.lpl[cell] : -INFINITY;
    const float pb = __expf(a + lpb + bn - lnP);
    const float pl = has_lab ? __expf(a + lpl + sv.beta[cell + 1] - lnP) : 0.f;
    const float g = grad_loss ? grad_loss[rc.b] : 1.f;
    const int lab = has_lab ? c.labels[(size_t)rc.b * U1 + rc.u + 1] : -1;
    const float G = g * (pb + pl);
    const float lgn = G != 0.f ? log2f(fabsf(G)) - sv.lnPD[cell] * kLog2e : -INFINITY;
    float dhb = G * __expf(lpb) - g * pb;
    const float dhl = has_lab ? G * __expf(lpl) - g * pl - (lab == c.sh.blank ? g * pb : 0.f)
                              : 0.f;
    if (has_lab && lab == c.sh.blank) dhb = dhl;
    const uint32_t bits = (uint32_t)(lab + 1) | (G < 0.f ? 0x80000000u : 0u);
    rec = make_float4(lgn, dhb, dhl, __uint_as_float(bits));
  }
  post[(long long)blockIdx.x * TILE + threadIdx.x] = rec;
}

// dh from the kept bf16 scores, in place (untiled mode: no recompute; Flash
// RNN-T blog, "Compute it, use it, make room"), from the same per-position
// records as the dh epilogue: dh_v = g (pb + pl) exp(h_v - lnPD)
// - g pb [v = blank] - g pl [v = label] (Eq. 10), as
// sign(g) exp2(h_v log2(e) + log2|g (pb + pl)| - lnPD log2(e)).  One block per
// tile; thread (k, s) owns the 8 consecutive columns of column group k
// (groups strided by the group width) for the rows s, s + S, s + 2S, ..., so
// a warp reads and writes 512 contiguous bytes of a row per access.  With
// dbO (16-byte aligned), each thread's column sums of the bf16 dh over its
// rows are added to it.
__global__ void __launch_bounds__(256)
k_dh_kept_bf16(ChunkArgs c, __nv_bfloat16* __restrict__ Hs, const float4* __restrict__ post,
               float* __restrict__ dbO, int groups) {
  // only the batch's tiles: the forward kept scores for exactly these
  if ((long long)blockIdx.x >= (long long)*c.sv.total_tiles - c.first_tile) return;
  const int V = c.sh.V, V8 = V / 8, blank = c.sh.blank;
  const int S = blockDim.x / groups, s0 = threadIdx.x / groups;
  __nv_bfloat16* tile = Hs + (long long)blockIdx.x * TILE * V;
  const float4* rec = post + (long long)blockIdx.x * TILE;
  const float2 l2 = make_float2(kLog2e, kLog2e);
  for (int k8 = threadIdx.x % groups; k8 < V8; k8 += groups) {
    const int v0 = 8 * k8;
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                     make_float2(0.f, 0.f)};
#pragma unroll 4
    for (int r = s0; r < TILE; r += S) {
      const DhState st = dh_state(__ldg(rec + r));
      uint4* hp = (uint4*)(tile + (long long)r * V + v0);
      const uint4 x = *hp;
      const float2 g2 = make_float2(st.lgn, st.lgn);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      float d[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 y = __ffma2_rn(make_float2(ptx::bf16lo(w[k]), ptx::bf16hi(w[k])), l2, g2);
        d[2 * k] = ptx::ex2(y.x);
        d[2 * k + 1] = ptx::ex2(y.y);
      }
      if (st.neg) {
#pragma unroll
        for (int j = 0; j < 8; ++j) d[j] = -d[j];
      }
      // the blank and label columns take their finished values (at most two
      // pieces of a row hold them)
      const int jb = blank - v0, jl = st.lab - v0;
      if ((unsigned)jb < 8u) {
#pragma unroll
        for (int j = 0; j < 8; ++j) d[j] = (j == jb) ? st.dhb : d[j];
      }
      if (st.lab >= 0 && (unsigned)jl < 8u) {
#pragma unroll
        for (int j = 0; j < 8; ++j) d[j] = (j == jl) ? st.dhl : d[j];
      }
      const uint4 o = pack8_bf16(d);
      *hp = o;
      const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        acc[k] = __fadd2_rn(acc[k], make_float2(ptx::bf16lo(ow[k]), ptx::bf16hi(ow[k])));
    }
    if (dbO) {
      ptx::red_add_v4(dbO + v0, acc[0].x, acc[0].y, acc[1].x, acc[1].y);
      ptx::red_add_v4(dbO + v0 + 4, acc[2].x, acc[2].y, acc[3].x, acc[3].y);
    }
  }
}

// The same pass streamed through shared memory (V <= 16384): a tile's kept
// scores are one contiguous range (128 rows x V bf16), which the block moves
// in chunks of whole rows (R rows, at most 32 KiB) through a ring of
// DHK_STAGES shared-memory buffers with 1-D bulk copies that one thread
// issues, so that many bytes are in flight with few registers.  dh is formed
// in place in shared memory (thread (k, s): column groups k, k + groups, ...
// of rows s, s + S, ... of the chunk; a warp touches 512 contiguous bytes)
// and the chunk is written back by a bulk store; a buffer is refilled once
// the store issued from it one chunk earlier has been read out.  The per-row
// terms are formed once per block from the posterior records.  Every wait is
// bounded: on a timeout the block sets RNNT_ERR_TIMEOUT, waits (bounded) for
// the copies it issued and leaves.
constexpr int DHK_STAGES = 3;
constexpr int DHK_CHUNK_MAX = 32768;
constexpr int DHK_GROUPS_MAX = 8;  // column groups a thread may own (V <= 256 * 8 * 8)

template <int NG>  // column groups a thread owns at most
__global__ void __launch_bounds__(256)
k_dh_kept_stream_bf16(ChunkArgs c, __nv_bfloat16* __restrict__ Hs,
                      const float4* __restrict__ post, float* __restrict__ dbO, int groups,
                      int R, int stage_bytes) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ uint64_t full[DHK_STAGES];
  __shared__ float4 rinfo[TILE];  // the rows' records (see k_posteriors)
  const long long have = (long long)*c.sv.total_tiles - c.first_tile;
  if ((long long)blockIdx.x >= have) return;
  const int V = c.sh.V, V8 = V / 8, blank = c.sh.blank;
  const int nchunks = TILE / R;
  const uint32_t cbytes = (uint32_t)R * (uint32_t)V * 2u;
  unsigned char* gtile = (unsigned char*)(Hs + (long long)blockIdx.x * TILE * V);
  const bool leader = threadIdx.x == 0;
  int issued = 0;
  if (leader) {
    for (int i = 0; i < DHK_STAGES; ++i) ptx::mbar_init(&full[i], 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (leader) {
    for (; issued < DHK_STAGES && issued < nchunks; ++issued) {
      ptx::mbar_arrive_expect_tx(&full[issued], cbytes);
      ptx::bulk_load(dsm + issued * stage_bytes, gtile + (size_t)issued * cbytes, cbytes,
                     &full[issued]);
    }
  }
  if (threadIdx.x < TILE)
    rinfo[threadIdx.x] = __ldg(post + (long long)blockIdx.x * TILE + threadIdx.x);
  __syncthreads();
  const int S = blockDim.x / groups, s0 = threadIdx.x / groups, k0 = threadIdx.x % groups;
  const float2 l2 = make_float2(kLog2e, kLog2e);
  float2 acc[NG][4];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[gi][k] = make_float2(0.f, 0.f);
  bool ok = true;
  int i = 0;
  for (; i < nchunks; ++i) {
    const int st = i % DHK_STAGES;
    bool got = ptx::mbar_wait(&full[st], (uint32_t)(i / DHK_STAGES) & 1u, WAIT_NS);
    if (got) {
      unsigned char* buf = dsm + st * stage_bytes;
      for (int r = s0; r < R; r += S) {
        const DhState st = dh_state(rinfo[i * R + r]);
        const float2 g2 = make_float2(st.lgn, st.lgn);
        const bool neg = st.neg;
        const int lab = st.lab;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
          const int k8 = k0 + gi * groups;
          if (k8 < V8) {
            uint4* pp = (uint4*)(buf + ((size_t)r * V8 + k8) * 16);
            const uint4 x = *pp;
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            float d[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 y =
                  __ffma2_rn(make_float2(ptx::bf16lo(w[k]), ptx::bf16hi(w[k])), l2, g2);
              d[2 * k] = ptx::ex2(y.x);
              d[2 * k + 1] = ptx::ex2(y.y);
            }
            if (neg) {
#pragma unroll
              for (int j = 0; j < 8; ++j) d[j] = -d[j];
            }
            // the blank and label columns take their finished values (at
            // most two pieces of a row hold them)
            const int jb = blank - 8 * k8, jl = lab - 8 * k8;
            if ((unsigned)jb < 8u) {
#pragma unroll
              for (int j = 0; j < 8; ++j) d[j] = (j == jb) ? st.dhb : d[j];
            }
            if (lab >= 0 && (unsigned)jl < 8u) {
#pragma unroll
              for (int j = 0; j < 8; ++j) d[j] = (j == jl) ? st.dhl : d[j];
            }
            const uint4 o = pack8_bf16(d);
            *pp = o;
            const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              acc[gi][k] =
                  __fadd2_rn(acc[gi][k], make_float2(ptx::bf16lo(ow[k]), ptx::bf16hi(ow[k])));
          }
        }
      }
      ptx::fence_proxy_async_smem();  // the dh writes are visible to the bulk store
    }
    if (!__syncthreads_and(got)) {
      ok = false;
      break;
    }
    if (leader) {
      ptx::bulk_store(gtile + (size_t)i * cbytes, dsm + st * stage_bytes, cbytes);
      ptx::bulk_commit();
      // refill the buffer of the previous chunk once its store has read it
      if (i >= 1 && issued < nchunks) {
        ptx::bulk_wait_read_1();
        const int rs = (i - 1) % DHK_STAGES;
        ptx::mbar_arrive_expect_tx(&full[rs], cbytes);
        ptx::bulk_load(dsm + rs * stage_bytes, gtile + (size_t)issued * cbytes, cbytes,
                       &full[rs]);
        ++issued;
      }
    }
  }
  if (leader) {
    if (!ok) {
      atomicOr(c.sv.status, status_bit(RNNT_ERR_TIMEOUT));
      // the loads issued and not consumed land before the block leaves
      for (int j = i; j < issued; ++j)
        ptx::mbar_wait(&full[j % DHK_STAGES], (uint32_t)(j / DHK_STAGES) & 1u, WAIT_NS);
    }
    ptx::bulk_wait_all();
  }
  if (ok && dbO) {
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      const int k8 = k0 + gi * groups;
      if (k8 < V8 && s0 < R) {
        ptx::red_add_v4(dbO + 8 * k8, acc[gi][0].x, acc[gi][0].y, acc[gi][1].x, acc[gi][1].y);
        ptx::red_add_v4(dbO + 8 * k8 + 4, acc[gi][2].x, acc[gi][2].y, acc[gi][3].x,
                        acc[gi][3].y);
      }
    }
  }
}

cudaError_t launch_dh_kept_bf16(const ChunkArgs& c, __nv_bfloat16* Hs, const float4* post,
                                float* dbO, cudaStream_t s) {
  // column groups: V/8 rounded up to whole warps, at most 256; row groups
  // fill the block up to 256 threads
  const int V = c.sh.V;
  const int groups = std::min(256, (int)cdiv(V / 8, 32) * 32);
  const int S = std::max(1, 256 / groups);
  const long long row_bytes = 2LL * V;
  const long long ng = cdiv(V / 8, groups);
  if (row_bytes <= DHK_CHUNK_MAX && ng <= DHK_GROUPS_MAX) {
    // rows per chunk: the largest power of two whose rows fit 16 KiB (at
    // least one row, at most the tile)
    int R = 1;
    while (R < TILE && 2 * R * row_bytes <= 16384) R *= 2;
    const int stage_bytes = (int)(((long long)R * row_bytes + 127) / 128 * 128);
    const int smem = DHK_STAGES * stage_bytes;
    auto kern = ng <= 1 ? k_dh_kept_stream_bf16<1>
                        : (ng <= 2 ? k_dh_kept_stream_bf16<2>
                                   : k_dh_kept_stream_bf16<DHK_GROUPS_MAX>);
    // dynamic plus static shared memory pass the 48 KiB default: opt in once
    // per instantiation to the largest ring
    static std::atomic<bool> opted[3][kDeviceSlots];
    std::atomic<bool>& done = opted[ng <= 1 ? 0 : (ng <= 2 ? 1 : 2)][device_slot()];
    if (!done.load()) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DHK_STAGES * DHK_CHUNK_MAX) != cudaSuccess)
        return cudaErrorInvalidValue;
      done.store(true);
    }
    kern<<<(unsigned)c.ntiles, groups * S, smem, s>>>(c, Hs, post, dbO, groups, R, stage_bytes);
    return cudaGetLastError();
  }
  k_dh_kept_bf16<<<(unsigned)c.ntiles, groups * S, 0, s>>>(c, Hs, post, dbO, groups);
  return cudaGetLastError();
}


// out[n] += sum over rows of an fp32 [R][N] matrix (N % 4 == 0).  A block is
// 8 row groups x 32 threads; each thread sums 4 consecutive columns (one
// 16-byte load per row), so a warp reads 512 contiguous bytes of a row.
__global__ void __launch_bounds__(256)
k_colsum_f32v(const float* __restrict__ X, long long R, int N, float* __restrict__ out,
              long long rows_per) {
  __shared__ float part[8][128];
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const int c0 = (blockIdx.x * 32 + lane) * 4;
  const long long r0 = (long long)blockIdx.y * rows_per;
  const long long r1 = min(R, r0 + rows_per);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c0 < N) {
    for (long long r = r0 + grp; r < r1; r += 8) {
      const float4 q = __ldg((const float4*)(X + r * N + c0));
      acc.x += q.x; acc.y += q.y; acc.z += q.z; acc.w += q.w;
    }
  }
  part[grp][lane * 4 + 0] = acc.x;
  part[grp][lane * 4 + 1] = acc.y;
  part[grp][lane * 4 + 2] = acc.z;
  part[grp][lane * 4 + 3] = acc.w;
  __syncthreads();
  if (threadIdx.x < 128) {
    const int c = blockIdx.x * 128 + threadIdx.x;
    if (c < N) {
      float sum = 0.f;
#pragma unroll
      for (int g = 0; g < 8; ++g) sum += part[g][threadIdx.x];
      if (sum != 0.f) atomicAdd(out + c, sum);
    }
  }
}

cudaError_t launch_colsum_f32v(const float* X, long long R, int N, float* out, cudaStream_t s) {
  if (R <= 0 || N <= 0) return cudaSuccess;
  if (N % 4 != 0) return launch_colsum(X, R, N, N, out, s);
  const int strips = (int)cdiv(N, 128);
  long long slabs = std::max<long long>(1, (long long)num_sms() * 4 / strips);
  long long rows_per = cdiv(R, slabs);
  if (cdiv(R, rows_per) > 65535) rows_per = cdiv(R, 65535);
  k_colsum_f32v<<<dim3(strips, (unsigned)cdiv(R, rows_per)), 256, 0, s>>>(X, R, N, out, rows_per);
  return cudaGetLastError();
}

// bf16 copy of an fp32 [R][N] matrix.
__global__ void k_f32_to_bf16(const float* __restrict__ x, __nv_bfloat16* __restrict__ y,
                              size_t n) {
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n; i += stride) y[i] = __float2bfloat16_rn(x[i]);
}

// Copy of a bf16 [B*P][N] matrix whose row (b, q) is kept iff q < len[b], else 0.
__global__ void k_mask_rows_bf16(const __nv_bfloat16* __restrict__ x,
                                 __nv_bfloat16* __restrict__ y, int B, int P, int N,
                                 const int32_t* __restrict__ len) {
  const size_t n = (size_t)B * P * N;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n; i += stride) {
    const size_t row = i / N;
    const int b = (int)(row / P), q = (int)(row % P);
    y[i] = (q < len[b]) ? x[i] : __float2bfloat16_rn(0.f);
  }
}

int elementwise_grid(size_t n) {
  size_t g = (n + 255) / 256;
  const size_t cap = (size_t)num_sms() * 16;
  return (int)std::max<size_t>(1, std::min(g, cap));
}

// Eight elements per thread step (two 16-byte loads, one 16-byte store).
__global__ void k_f32_to_bf16_x8(const float4* __restrict__ x, uint4* __restrict__ y,
                                 size_t n8) {
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n8; i += stride) {
    const float4 a = __ldg(x + 2 * i), b = __ldg(x + 2 * i + 1);
    y[i] = make_uint4(ptx::pack_bf16x2(a.x, a.y), ptx::pack_bf16x2(a.z, a.w),
                      ptx::pack_bf16x2(b.x, b.y), ptx::pack_bf16x2(b.z, b.w));
  }
}

// y = bf16(x), n elements (16-byte aligned pointers: eight per step).
cudaError_t launch_f32_to_bf16(const float* x, __nv_bfloat16* y, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if ((((uintptr_t)x | (uintptr_t)y) & 15) != 0) {
    k_f32_to_bf16<<<elementwise_grid(n), 256, 0, s>>>(x, y, n);
    return cudaGetLastError();
  }
  const size_t n8 = n / 8, tail = n % 8;
  if (n8)
    k_f32_to_bf16_x8<<<elementwise_grid(n8), 256, 0, s>>>((const float4*)x, (uint4*)y, n8);
  if (tail) k_f32_to_bf16<<<1, 32, 0, s>>>(x + 8 * n8, y + 8 * n8, tail);
  return cudaGetLastError();
}

// k_mask_rows_bf16 with rows of N8 16-byte words: a warp per row (one
// division per row, not per element).
__global__ void k_mask_rows_bf16_x8(const uint4* __restrict__ x, uint4* __restrict__ y,
                                    long long rows, int P, int N8,
                                    const int32_t* __restrict__ len) {
  const int lane = threadIdx.x & 31;
  const long long w0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r = w0; r < rows; r += nw) {
    const int b = (int)(r / P), q = (int)(r - (long long)b * P);
    const bool keep = q < __ldg(len + b);
    const uint4* xs = x + r * N8;
    uint4* ys = y + r * N8;
    for (int k = lane; k < N8; k += 32) ys[k] = keep ? __ldg(xs + k) : make_uint4(0, 0, 0, 0);
  }
}

// y[b,q,:] = x[b,q,:] for q < len[b], else 0 (B x P rows of N bf16).
cudaError_t launch_mask_rows_bf16(const __nv_bfloat16* x, __nv_bfloat16* y, int B, int P, int N,
                                  const int32_t* len, cudaStream_t s) {
  const long long rows = (long long)B * P;
  if (rows == 0 || N == 0) return cudaSuccess;
  if ((N & 7) != 0 || (((uintptr_t)x | (uintptr_t)y) & 15) != 0) {
    k_mask_rows_bf16<<<elementwise_grid((size_t)rows * N), 256, 0, s>>>(x, y, B, P, N, len);
    return cudaGetLastError();
  }
  const int grid = (int)std::max<long long>(
      1, std::min<long long>((rows + 7) / 8, (long long)num_sms() * 16));
  k_mask_rows_bf16_x8<<<grid, 256, 0, s>>>((const uint4*)x, (uint4*)y, rows, P, N / 8, len);
  return cudaGetLastError();
}

// ---- tensor maps ----------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  });
  return fn;
}

// Row-major matrix [rows][cols] (cols contiguous) of bf16 (e8 = false; box
// 64 x box_rows) or of one-byte e4m3 values (e8 = true; box 128 x box_rows):
// 128 bytes of a row per box line, 128-byte swizzle, zero fill outside the
// matrix.
bool make_tmap(CUtensorMap* m, const void* ptr, long long rows, long long cols, int box_rows,
               bool e8 = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * (e8 ? 1 : 2)};
  cuuint32_t box[2] = {e8 ? 128u : 64u, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, e8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Store map of a row-major bf16 matrix [rows][cols]: 32 x 32 boxes (one
// epilogue warp's block), 64-byte swizzle.
bool make_tmap_store32(CUtensorMap* m, const void* ptr, long long rows, long long cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// One GEMM: C-shaped problem M x N x K with A = [M][K] (a_mn = 0) or [K][M]
// (a_mn = 1) and B = [N][K] (b_mn = 0) or [K][N] (b_mn = 1), all bf16.
struct GemmDesc {
  const void* A;
  int a_mn;
  const void* B;
  int b_mn;
  int M, N, K;
  int e8;  // A and B are e4m3 (one byte per element, K-major), else bf16
};

template <int BN, int AMN, int BMN, int EPI, int F8 = 0>
cudaError_t launch_gemm_t(const GemmDesc& g, TcParams p, cudaStream_t s) {
  using C = Cfg<BN, EPI>;
  auto kern = k_tc_gemm<BN, AMN, BMN, EPI, F8>;
  CUtensorMap ta, tb;
  const bool ok_a = AMN ? make_tmap(&ta, g.A, g.K, g.M, 64)
                        : make_tmap(&ta, g.A, g.M, g.K, BM, F8 != 0);
  const bool ok_b = BMN ? make_tmap(&tb, g.B, g.K, g.N, 64)
                        : make_tmap(&tb, g.B, g.N, g.K, BN, F8 != 0);
  if (!ok_a || !ok_b) return cudaErrorInvalidValue;
  // dh / kept-score epilogues: the store map of the [M][N] tile buffer; the
  // other epilogues never read the third map
  CUtensorMap tc = ta;
  if (box_store(EPI) && !make_tmap_store32(&tc, p.Hout, g.M, g.N)) return cudaErrorInvalidValue;
  static std::atomic<bool> opted_in[kDeviceSlots];  // per instantiation and device
  std::atomic<bool>& opted = opted_in[device_slot()];
  if (!opted.load()) {
    // up to the per-block maximum: the score epilogues' bias copy goes behind
    // the kernel's own layout when it fits
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    opted.store(true);
  }
  int smem_bytes = C::SMEM;
  p.sbias = 0;
  if ((lse_like(EPI) || EPI == EPI_DH) && p.bias && g.N % 8 == 0 &&
      C::SMEM + 2 * g.N <= SMEM_LIMIT) {
    p.sbias = 1;
    smem_bytes = C::SMEM + 2 * g.N;
  }
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.m_tiles = (int)cdiv(g.M, BM);
  p.n_tiles = (int)cdiv(g.N, BN);
  p.kb_total = (int)cdiv(g.K, F8 ? 128 : BK);
  if (p.k_splits < 1) p.k_splits = 1;
  p.kb_per_split = (int)cdiv(p.kb_total, p.k_splits);
  p.k_splits = (int)cdiv(p.kb_total, p.kb_per_split);
  if (p.n_split < 1 || !p.row_complete) p.n_split = 1;
  if (p.n_split > p.n_tiles) p.n_split = p.n_tiles;
  p.units = p.row_complete ? p.m_tiles * p.n_split : p.m_tiles * p.n_tiles * p.k_splits;
  if (p.units <= 0 || g.K <= 0) return cudaSuccess;
  // persistent: at most one CTA per SM, each walking units gridDim apart
  const int grid = std::min(p.units, num_sms());
  // programmatic dependent launch: the kernel's set-up (barriers, TMEM,
  // descriptor prefetch) may overlap the tail of the stream's previous kernel
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, p);
}

template <int EPI>
cudaError_t launch_gemm(const GemmDesc& g, const TcParams& p, int bn, cudaStream_t s) {
  // Only the operand layouts each epilogue is used with are instantiated:
  // the lattice epilogues take K-major scores/z (and an MN-major W^O for
  // dz); the store and atomic epilogues take every layout.
  if constexpr (lse_like(EPI) || EPI == EPI_DH) {
    if (g.a_mn || g.b_mn) return cudaErrorInvalidValue;
    if (g.e8) {  // e4m3 scores: 256-wide N tiles (one W^O scale block each)
      if (bn != 256) return cudaErrorInvalidValue;
      return launch_gemm_t<256, 0, 0, EPI, 1>(g, p, s);
    }
    if (bn == 256) return launch_gemm_t<256, 0, 0, EPI>(g, p, s);
    return launch_gemm_t<128, 0, 0, EPI>(g, p, s);
  } else if constexpr (EPI == EPI_DA) {
    if (g.a_mn || !g.b_mn) return cudaErrorInvalidValue;
    if (bn == 256) return launch_gemm_t<256, 0, 1, EPI>(g, p, s);
    return launch_gemm_t<128, 0, 1, EPI>(g, p, s);
  } else {
    const int code = (bn == 256 ? 4 : 0) | (g.a_mn ? 2 : 0) | (g.b_mn ? 1 : 0);
    switch (code) {
      case 0: return launch_gemm_t<128, 0, 0, EPI>(g, p, s);
      case 1: return launch_gemm_t<128, 0, 1, EPI>(g, p, s);
      case 2: return launch_gemm_t<128, 1, 0, EPI>(g, p, s);
      case 3: return launch_gemm_t<128, 1, 1, EPI>(g, p, s);
      case 4: return launch_gemm_t<256, 0, 0, EPI>(g, p, s);
      case 5: return launch_gemm_t<256, 0, 1, EPI>(g, p, s);
      case 6: return launch_gemm_t<256, 1, 0, EPI>(g, p, s);
      default: return launch_gemm_t<256, 1, 1, EPI>(g, p, s);
    }
  }
}

int pick_bn(int N, long long M = 1LL << 40) {
  // the tile width that wastes the fewest MMA columns (ties: the wider one),
  // unless 256-wide tiles leave more than half of the SMs without a tile
  const long long w256 = cdiv(N, 256) * 256, w128 = cdiv(N, 128) * 128;
  if (cdiv(M, BM) * cdiv(N, 256) < num_sms() / 2) return 128;
  return w256 <= w128 ? 256 : 128;
}

// Split K into s ranges (>= 8 K blocks each) so that units_mn * s CTAs fill
// whole waves of SMs; a small penalty per split keeps the atomics down.
int pick_splits(int units_mn, int K) {
  const int kb = (int)cdiv(K, BK);
  const int smax = std::max(1, kb / 8);
  int best = 1;
  double best_score = -1.0;
  for (int sp = 1; sp <= smax && sp <= 64; ++sp) {
    const long long units = (long long)units_mn * sp;
    const long long waves = cdiv(units, num_sms());
    const double eff = (double)units / (double)(waves * num_sms());
    const double score = eff - 0.004 * sp;
    if (score > best_score + 1e-9) { best_score = score; best = sp; }
  }
  return best;
}

#define TC_CHECK(expr)                                   \
  do {                                                   \
    cudaError_t e_ = (expr);                             \
    if (e_ != cudaSuccess) return e_;                    \
  } while (0)

}  // namespace

// ===========================================================================
// Entry points used by the C ABI (tc.h).

rnnt_status tc_check_shape(const Plan& p) {
  if (p.H % 8 || p.V % 8 || p.HA % 8 || p.HL % 8) return RNNT_ERR_UNSUPPORTED_SHAPE;
  // e4m3 rows of H bytes: TMA strides are multiples of 16 bytes
  if (p.f8 && p.H % 16) return RNNT_ERR_UNSUPPORTED_SHAPE;
  if (!encode_fn()) return RNNT_ERR_CUDA;
  return RNNT_OK;
}

cudaError_t tc_projection(const Plan& p, const void* X, const void* W, const void* bias, int M,
                          int K, float* out, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  ProfScope ps("tc_projection", s);
  GemmDesc g{X, 0, W, 0, M, p.H, K};
  TcParams tp{};
  tp.C = out;
  tp.ldc = p.H;
  tp.bias = (const __nv_bfloat16*)bias;
  return launch_gemm<EPI_STORE>(g, tp, pick_bn(p.H, M), s);
}

cudaError_t tc_quantize_wo(const Plan& p, const void* WO, void* wo8, void* wodq, float* nscale,
                           cudaStream_t s) {
  return launch_quantize_wo(WO, wo8, wodq, nscale, p.V, p.H, s);
}

rnnt_status tc_forward_tiles(const Plan& p, const SavedView& sv, const rnnt_params* pr,
                             const int32_t* labels, const int32_t* T_len, const int32_t* U_len,
                             const float* pA, const float* pL, void* Zv, void* Hkeep,
                             const TcF8* f8, cudaStream_t s) {
  __nv_bfloat16* Z = (__nv_bfloat16*)Zv;
  if (!Z) return RNNT_ERR_INVALID_ARG;
  long long nch = 0;
  rnnt_status st = chunk_count(p, sv, s, &nch);
  if (st != RNNT_OK) return st;
  for (long long k = 0; k < nch; ++k) {
    ChunkArgs c = chunk_args(p, sv, k, labels, T_len, U_len);
    {
      // e4m3 scores: their operand only (and the bf16 z that untiled mode
      // keeps for the backward)
      ProfScope ps("tc_build_z", s);
      if (launch_build_z_bf16(c, pA, pL, (f8 && !Hkeep) ? nullptr : Z, f8 ? f8->z8 : nullptr,
                              s) != cudaSuccess)
        return RNNT_ERR_CUDA;
    }
    ProfScope ps("tc_fwd_tiles", s);
    GemmDesc g{Z, 0, pr->WO, 0, (int)p.chunk_rows, p.V, p.H};
    TcParams tp{};
    if (f8) {
      g.A = f8->z8;
      g.B = f8->wo8;
      g.e8 = 1;
      tp.nscale = f8->nscale;
    }
    tp.row_complete = 1;
    tp.bias = (const __nv_bfloat16*)pr->bO;
    tp.ch = c;
    tp.Hout = (__nv_bfloat16*)Hkeep;
    tp.status = sv.status;
    tp.tiles_on = TILES_ON_M;
    const cudaError_t e = Hkeep ? launch_gemm<EPI_LSEK>(g, tp, 256, s)
                                : launch_gemm<EPI_LSE>(g, tp, 256, s);
    if (e != cudaSuccess) return RNNT_ERR_CUDA;
  }
  return RNNT_OK;
}

rnnt_status tc_backward_tiles(const Plan& p, const SavedView& sv, const rnnt_params* pr,
                              const int32_t* labels, const int32_t* T_len, const int32_t* U_len,
                              const float* grad_loss, const float* pA, const float* pL, void* Zv,
                              void* Hv, bool untiled, bool z_resident, float* dA, float* dLr,
                              float* dWO,
                              float* dbO, float4* post, const TcF8* f8, const PreLaunch* pre,
                              const PreLaunch* after, cudaStream_t s) {
  __nv_bfloat16* Z = (__nv_bfloat16*)Zv;
  __nv_bfloat16* Hs = (__nv_bfloat16*)Hv;
  long long nch = 0;
  rnnt_status st = chunk_count(p, sv, s, &nch);
  if (st != RNNT_OK) return st;
  const int rows = (int)p.chunk_rows;
  if (pre && (untiled || nch == 0)) {
    st = (*pre)(s);
    if (st != RNNT_OK) return st;
  }
  if (nch == 0 && after) return (*after)(s);
  for (long long k = 0; k < nch; ++k) {
    ChunkArgs c = chunk_args(p, sv, k, labels, T_len, U_len);
    if (!untiled) {
      {
        // the z rebuild, the posterior records and (first chunk) the caller's
        // preparatory launches are independent of one another
        Fork fork(s, 2);
        if (k == 0 && pre) {
          st = (*pre)(fork.side(1));
          if (st != RNNT_OK) return st;
        }
        {
          ProfScope ps("tc_posteriors", fork.side(0));
          k_posteriors<<<(unsigned)c.ntiles, TILE, 0, fork.side(0)>>>(c, grad_loss, post);
          if (cudaGetLastError() != cudaSuccess) return RNNT_ERR_CUDA;
        }
        // (e4m3 scores: the forward kept only the e4m3 rows; both are built)
        if (!(z_resident && nch == 1) || f8) {
          ProfScope ps("tc_build_z", s);
          if (launch_build_z_bf16(c, pA, pL, Z, f8 ? f8->z8 : nullptr, s) != cudaSuccess)
            return RNNT_ERR_CUDA;
        }
        if (fork.join() != cudaSuccess) return RNNT_ERR_CUDA;
      }
      // recompute the tile's scores and overwrite them with dh
      ProfScope ps("tc_bwd_dh", s);
      GemmDesc g{Z, 0, pr->WO, 0, rows, p.V, p.H};
      TcParams tp{};
      if (f8) {  // the scores recomputed exactly as the forward formed them
        g.A = f8->z8;
        g.B = f8->wo8;
        g.e8 = 1;
        tp.nscale = f8->nscale;
      }
      tp.row_complete = 1;
      tp.bias = (const __nv_bfloat16*)pr->bO;
      tp.ch = c;
      tp.grad_loss = grad_loss;
      tp.Hout = Hs;
      tp.post = post;
      // each tile's V range split over up to 4 units, the kernel choosing
      // from the batch's tile count
      tp.n_split = 4;
      tp.n_split_auto = 1;
      tp.status = sv.status;
      // db^O: column sums of dh formed in the same epilogue (into a 16-byte
      // aligned workspace vector)
      tp.dbO = dbO;
      tp.tiles_on = TILES_ON_M;
      if (launch_gemm<EPI_DH>(g, tp, 256, s) != cudaSuccess) return RNNT_ERR_CUDA;
    } else {
      {
        ProfScope ps("tc_posteriors", s);
        k_posteriors<<<(unsigned)c.ntiles, TILE, 0, s>>>(c, grad_loss, post);
        if (cudaGetLastError() != cudaSuccess) return RNNT_ERR_CUDA;
      }
      // dh over the kept scores, db^O in the same pass
      ProfScope ps("tc_dh_kept", s);
      if (launch_dh_kept_bf16(c, Hs, post, dbO, s) != cudaSuccess) return RNNT_ERR_CUDA;
    }
    {  // dz = dh W^O, da = dz (1 - z^2) reduced into dA and dLr
      ProfScope ps("tc_bwd_dz", s);
      // (e4m3 scores: the dequantized W^O_q the scores were formed with)
      GemmDesc g{Hs, 0, f8 ? f8->wodq : pr->WO, 1, rows, p.H, p.V};
      TcParams tp{};
      tp.ch = c;
      tp.Zin = Z;
      tp.dA = dA;
      tp.dLr = dLr;
      tp.status = sv.status;
      tp.tiles_on = TILES_ON_M;
      if (launch_gemm<EPI_DA>(g, tp, pick_bn(p.H, rows), s) != cudaSuccess)
        return RNNT_ERR_CUDA;
    }
    // the last chunk's dW^O runs beside the caller's work that needs only
    // dA and dLr (the encoder-side gradients)
    const bool last = k + 1 == nch;
    Fork fork(s, last && after && dWO ? 1 : 0);
    if (dWO) {  // dW^O += dh^T z, split over the chunk's rows
      ProfScope ps("tc_bwd_dwo", fork.side(0));
      GemmDesc g{Hs, 1, Z, 1, p.V, p.H, rows};
      TcParams tp{};
      const int bn = pick_bn(p.H);
      tp.k_splits = pick_splits((int)(cdiv(p.V, BM) * cdiv(p.H, bn)), rows);
      tp.C = dWO;
      tp.ldc = p.H;
      tp.status = sv.status;
      tp.ch = c;
      tp.tiles_on = TILES_ON_K;
      if (launch_gemm<EPI_ATOMIC>(g, tp, bn, fork.side(0)) != cudaSuccess)
        return RNNT_ERR_CUDA;
    }
    if (last && after) {
      st = (*after)(s);
      if (st != RNNT_OK) return st;
    }
    if (fork.join() != cudaSuccess) return RNNT_ERR_CUDA;
  }
  return RNNT_OK;
}

rnnt_status tc_encoder_grads(const Plan& p, char* ws, const void* hA, const void* hL,
                             const rnnt_params* pr, const int32_t* Teff, const int32_t* Ueff,
                             float* dA, float* dLr, void* dhA, void* dhL, float* dWA,
                             float* dWL, float* dbZ, const EncOut& out, cudaStream_t s) {
  // the bf16 operands of the encoder GEMMs go straight into the caller's
  // hand-off buffers when those are bf16
  __nv_bfloat16* dA16 = (out.bf16 && out.dA) ? (__nv_bfloat16*)out.dA
                                             : (__nv_bfloat16*)(ws + p.w_dA16);
  __nv_bfloat16* dLr16 = (out.bf16 && out.dL) ? (__nv_bfloat16*)out.dL
                                              : (__nv_bfloat16*)(ws + p.w_dLr16);
  __nv_bfloat16* hAm = (__nv_bfloat16*)(ws + p.w_hAm);
  __nv_bfloat16* hLm = (__nv_bfloat16*)(ws + p.w_hLm);
  const size_t nA = (size_t)p.B * p.T * p.H, nL = (size_t)p.B * p.U1 * p.H;
  // Two phases of independent launches, each spread over side streams: the
  // bf16 operands, then the four encoder-side GEMMs and db^Z.
  {
    ProfScope ps("tc_enc_prep", s);
    ps.set_kernels(2 + (dWA ? 1 : 0) + (dWL ? 1 : 0));
    Fork fork(s, 3);
    if (launch_f32_to_bf16(dA, dA16, nA, s) != cudaSuccess ||
        launch_f32_to_bf16(dLr, dLr16, nL, fork.side(0)) != cudaSuccess)
      return RNNT_ERR_CUDA;
    if (dWA && launch_mask_rows_bf16((const __nv_bfloat16*)hA, hAm, p.B, p.T, p.HA, Teff,
                                     fork.side(1)) != cudaSuccess)
      return RNNT_ERR_CUDA;
    if (dWL && launch_mask_rows_bf16((const __nv_bfloat16*)hL, hLm, p.B, p.U1, p.HL, Ueff,
                                     fork.side(2)) != cudaSuccess)
      return RNNT_ERR_CUDA;
    // fp32 hand-off: the accumulators themselves
    if (!out.bf16 && out.dA &&
        cudaMemcpyAsync(out.dA, dA, nA * sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return RNNT_ERR_CUDA;
    if (!out.bf16 && out.dL &&
        cudaMemcpyAsync(out.dL, dLr, nL * sizeof(float), cudaMemcpyDeviceToDevice,
                        fork.side(0)) != cudaSuccess)
      return RNNT_ERR_CUDA;
    if (fork.join() != cudaSuccess) return RNNT_ERR_CUDA;
  }
  ProfScope ps("tc_enc_grads", s);
  ps.set_kernels((dhA ? 1 : 0) + (dhL ? 1 : 0) + (dWA ? 1 : 0) + (dWL ? 1 : 0) + (dbZ ? 1 : 0));
  Fork fork(s, 3);
  const int MA = p.B * p.T, ML = p.B * p.U1;
  if (dWA) {  // dW^A = dA^T hA: A = dA16 as [K=MA][M=H], B = hAm as [K=MA][N=HA]
    GemmDesc g{dA16, 1, hAm, 1, p.H, p.HA, MA};
    TcParams tp{};
    const int bn = pick_bn(p.HA);
    tp.k_splits = pick_splits((int)(cdiv(p.H, BM) * cdiv(p.HA, bn)), MA);
    tp.C = dWA;
    tp.ldc = p.HA;
    if (launch_gemm<EPI_ATOMIC>(g, tp, bn, s) != cudaSuccess) return RNNT_ERR_CUDA;
  }
  if (dhA) {  // dh^A = dA W^A: A = dA16 [MA][H], B = W^A [H][HA] (K rows, N contiguous)
    GemmDesc g{dA16, 0, pr->WA, 1, MA, p.HA, p.H};
    TcParams tp{};
    if (out.bf16) tp.Cb = (__nv_bfloat16*)dhA;
    else tp.C = (float*)dhA;
    tp.ldc = p.HA;
    if (launch_gemm<EPI_STORE>(g, tp, pick_bn(p.HA, MA), fork.side(0)) != cudaSuccess)
      return RNNT_ERR_CUDA;
  }
  if (dhL) {
    GemmDesc g{dLr16, 0, pr->WL, 1, ML, p.HL, p.H};
    TcParams tp{};
    if (out.bf16) tp.Cb = (__nv_bfloat16*)dhL;
    else tp.C = (float*)dhL;
    tp.ldc = p.HL;
    if (launch_gemm<EPI_STORE>(g, tp, pick_bn(p.HL, ML), fork.side(1)) != cudaSuccess)
      return RNNT_ERR_CUDA;
  }
  if (dWL) {
    GemmDesc g{dLr16, 1, hLm, 1, p.H, p.HL, ML};
    TcParams tp{};
    const int bn = pick_bn(p.HL);
    tp.k_splits = pick_splits((int)(cdiv(p.H, BM) * cdiv(p.HL, bn)), ML);
    tp.C = dWL;
    tp.ldc = p.HL;
    if (launch_gemm<EPI_ATOMIC>(g, tp, bn, fork.side(2)) != cudaSuccess)
      return RNNT_ERR_CUDA;
  }
  if (dbZ) {  // db^Z = sum of dA over frames (= sum of da over every position)
    if (launch_colsum_f32v(dA, (long long)p.B * p.T, p.H, dbZ, fork.side(1)) != cudaSuccess)
      return RNNT_ERR_CUDA;
  }
  if (fork.join() != cudaSuccess) return RNNT_ERR_CUDA;
  return RNNT_OK;
}

}  // namespace rnnt

// ===========================================================================
// Test hook (include/rnnt_testing.h): the GEMM with its first pipeline stage
// never filled, so the MMA thread's bounded wait runs out.
extern "C" rnnt_status rnnt_testing_gemm_timeout(int M, int N, int K, const void* A,
                                                 const void* B, float* C, int32_t* status,
                                                 unsigned long long wait_ns, void* stream) {
  using namespace rnnt;
  if (M <= 0 || N <= 0 || K <= 0 || !A || !B || !C || !status || wait_ns == 0)
    return RNNT_ERR_INVALID_ARG;
  if (K % 8) return RNNT_ERR_UNSUPPORTED_SHAPE;
  if (!encode_fn()) return RNNT_ERR_CUDA;
  GemmDesc g{A, 0, B, 0, M, N, K};
  TcParams tp{};
  tp.C = C;
  tp.ldc = N;
  tp.status = status;
  tp.wait_ns = wait_ns;
  tp.skip_first_fill = 1;
  cudaError_t e = launch_gemm<EPI_STORE>(g, tp, 128, (cudaStream_t)stream);
  return e == cudaSuccess ? RNNT_OK : RNNT_ERR_CUDA;
}

// ===========================================================================
// Test hook (include/rnnt_testing.h): one raw GEMM through the same kernel.
extern "C" rnnt_status rnnt_testing_gemm_bf16(int M, int N, int K, const void* A, int a_mn,
                                              const void* B, int b_mn, float* C, int accumulate,
                                              int k_splits, int bn, void* stream) {
  using namespace rnnt;
  if (M <= 0 || N <= 0 || K <= 0 || !A || !B || !C) return RNNT_ERR_INVALID_ARG;
  if ((a_mn ? M : K) % 8 || (b_mn ? N : K) % 8) return RNNT_ERR_UNSUPPORTED_SHAPE;
  if (bn != 128 && bn != 256) return RNNT_ERR_INVALID_ARG;
  if (!encode_fn()) return RNNT_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  GemmDesc g{A, a_mn, B, b_mn, M, N, K};
  TcParams tp{};
  tp.C = C;
  tp.ldc = N;
  tp.k_splits = k_splits;
  cudaError_t e = accumulate ? launch_gemm<EPI_ATOMIC>(g, tp, bn, s)
                             : launch_gemm<EPI_STORE>(g, tp, bn, s);
  return e == cudaSuccess ? RNNT_OK : RNNT_ERR_CUDA;
}

// ===========================================================================
// Test hook (include/rnnt_testing.h): the W^O quantization of the e4m3 scores.
extern "C" rnnt_status rnnt_testing_quantize_wo(int V, int H, const void* WO, void* Q, void* Wdq,
                                                float* nscale, void* stream) {
  using namespace rnnt;
  if (V <= 0 || H <= 0 || (H & 1) || !WO || !Q || !Wdq || !nscale) return RNNT_ERR_INVALID_ARG;
  return launch_quantize_wo(WO, Q, Wdq, nscale, V, H, (cudaStream_t)stream) == cudaSuccess
             ? RNNT_OK
             : RNNT_ERR_CUDA;
}
