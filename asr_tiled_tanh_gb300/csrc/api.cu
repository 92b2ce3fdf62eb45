// api.cu -- the C ABI of librnnt_gb300 (declared in include/rnnt.h).
//
// Host side only: argument checks, the layout of the caller's `saved` and
// `ws` buffers, and the order of kernel launches on the caller's stream.
// Every arithmetic step runs in this library's CUDA kernels.
//
// Forward (Flash RNN-T blog, "Compute it, use it, make room"; sample-wise
// transducer paper §2):
//   1. validate lengths/labels, per-sample tile counts and offsets;
//   2. joint projections pA = hA W^A^T + b^Z, pL = hL W^L^T (the matrix
//      products of Eq. 3 hoisted out of the lattice: they depend on t or u
//      only);
//   3. per tile: z = tanh(pA[t] + pL[u]), scores h = W^O z + b^O, and from
//      the scores only ln P_D and the blank/label log-probabilities (Eq. 7);
//   4. alpha/beta and the loss (Eq. 8-9).
// Backward (Flash RNN-T: recompute each tile, overwrite its scores with their
// gradients; sample-wise paper §4: accumulate the parameter gradients):
//   per tile: recompute z and h, dh in place (Eq. 10), dz = dh W^O,
//   da = dz (1 - z^2) summed over u into dA[b,t] and over t into dLr[b,u],
//   dW^O += dh^T z, db^O += sum dh; then dh^A = dA W^A, dW^A = dA^T hA,
//   dh^L = dLr W^L, dW^L = dLr^T hL, db^Z = sum dA.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "kernels.h"
#include "profile.h"
#include "streams.h"
#include "tc.h"

using namespace rnnt;

namespace {

constexpr long long kMaxI32 = 2147483647LL;

bool make_plan(const rnnt_dims* d, Plan* p) {
  if (!d) return false;
  if (d->B < 0 || d->T < 1 || d->U1 < 1 || d->HA < 1 || d->HL < 1 || d->H < 1 || d->V < 1)
    return false;
  if (d->blank < 0 || d->blank >= d->V) return false;
  if (d->dtype != RNNT_F32 && d->dtype != RNNT_BF16 && d->dtype != RNNT_BF16_E4M3) return false;
  if (d->mode != RNNT_TILED && d->mode != RNNT_UNTILED) return false;
  if (d->tile_cells < 0) return false;
  std::memset(p, 0, sizeof(*p));
  p->B = d->B; p->T = d->T; p->U1 = d->U1; p->HA = d->HA; p->HL = d->HL; p->H = d->H;
  p->V = d->V; p->blank = d->blank; p->dtype = d->dtype; p->mode = d->mode;
  p->tc = d->dtype == RNNT_BF16 || d->dtype == RNNT_BF16_E4M3;  // bf16 inputs: tensor cores
  p->f8 = p->tc && d->dtype == RNNT_BF16_E4M3;
  p->max_tiles = (long long)d->B * cdiv(d->T, TT) * cdiv(d->U1, TU);
  if (p->max_tiles > kMaxI32 / TILE) return false;
  if ((long long)d->B * d->T * d->U1 > kMaxI32 * 8LL) return false;
  p->zelem = p->tc ? 2 : 4;
  p->helem = p->tc ? 2 : 4;
  const size_t B = d->B, T = d->T, U1 = d->U1, H = d->H, V = d->V, HA = d->HA, HL = d->HL;
  if (d->mode == RNNT_UNTILED) {
    p->chunk_tiles = p->max_tiles;
  } else {
    long long ct;
    if (d->tile_cells > 0) {
      ct = cdiv(d->tile_cells, TILE);
    } else {
      // default: at most 2 GiB of tile buffers, in whole waves of 152 tiles
      const long long per_tile = (long long)TILE * (H * p->zelem + V * p->helem);
      ct = (2048LL << 20) / per_tile;
      ct = ct / 152 * 152;
      if (ct < 152) ct = 152;
    }
    p->chunk_tiles = ct < p->max_tiles ? ct : p->max_tiles;
  }
  if (p->chunk_tiles < 1) p->chunk_tiles = 1;
  p->chunk_rows = p->chunk_tiles * TILE;
  const size_t rows = (size_t)p->chunk_rows;

  size_t o = 0;
  auto put = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
  p->s_status = put(sizeof(SavedHeader));
  p->s_prefix = put(4 * (B + 1));
  p->s_tiles = put(16 * (size_t)(p->max_tiles ? p->max_tiles : 1));
  p->s_lnP = put(4 * (B ? B : 1));
  const size_t ncell = B * T * U1;
  p->s_lpb = put(4 * ncell);
  p->s_lpl = put(4 * ncell);
  p->s_lnPD = put(4 * ncell);
  p->s_alpha = put(4 * ncell);
  p->s_beta = put(4 * ncell);
  // the joint projections are kept for the backward (tiled mode recomputes z from them)
  p->s_pA = put(4 * B * T * H);
  p->s_pL = put(4 * B * U1 * H);
  if (d->mode == RNNT_UNTILED) {
    p->s_z = put(rows * H * p->zelem);
    p->s_h = put(rows * V * p->helem);
  }
  p->s_total = o;

  o = 0;
  p->w_dA = put(4 * B * T * H);
  p->w_dLr = put(4 * B * U1 * H);
  if (d->mode == RNNT_TILED) {
    p->w_z = put(rows * H * p->zelem);
    p->w_h = put(rows * V * p->helem);
  }
  if (!p->tc) {
    p->w_dz = put(4 * rows * H);
  } else {
    p->w_post = put(16 * rows);
    p->w_dA16 = put(2 * B * T * H);
    p->w_dLr16 = put(2 * B * U1 * H);
    p->w_hAm = put(2 * B * T * HA);
    p->w_hLm = put(2 * B * U1 * HL);
    p->w_dbO = put(4 * V);  // db^O accumulated here (16-byte aligned), then copied out
  }
  if (p->f8) {
    p->w_z8 = put(rows * H);              // e4m3(2^8 z) rows of a chunk
    p->w_wo8 = put(V * H);                // W^O in e4m3, per 256-row block scales
    p->w_wodq = put(2 * V * H);           // the dequantized W^O_q, bf16
    p->w_nscale = put(4 * ((V + 255) / 256));
  }
  p->w_len = put(8 * (B ? B : 1));  // effective lengths of accepted samples (2 x int32 [B])
  p->w_total = o;
  return true;
}

SavedView saved_view(const Plan& p, void* saved) {
  char* s = (char*)saved;
  SavedView v;
  SavedHeader* hdr = (SavedHeader*)(s + p.s_status);
  v.status = &hdr->status;
  v.total_tiles = &hdr->total_tiles;
  v.prefix = (int32_t*)(s + p.s_prefix);
  v.tiles = (int4*)(s + p.s_tiles);
  v.lnP = (float*)(s + p.s_lnP);
  v.lpb = (float*)(s + p.s_lpb);
  v.lpl = (float*)(s + p.s_lpl);
  v.lnPD = (float*)(s + p.s_lnPD);
  v.alpha = (float*)(s + p.s_alpha);
  v.beta = (float*)(s + p.s_beta);
  return v;
}

Shape shape_of(const Plan& p) { return Shape{p.B, p.T, p.U1, p.H, p.V, p.blank}; }

bool aligned(const void* x) { return ((uintptr_t)x & (ALIGN - 1)) == 0; }
// (NULL counts as aligned: optional arrays)
bool aligned16(const void* x) { return ((uintptr_t)x & 15) == 0; }

#define RNNT_CHECK(expr)                               \
  do {                                                 \
    cudaError_t e_ = (expr);                           \
    if (e_ != cudaSuccess) {                           \
      if (getenv("RNNT_VERBOSE"))                      \
        fprintf(stderr, "rnnt: %s -> %s (%s:%d)\n", #expr, cudaGetErrorString(e_), \
                __FILE__, __LINE__);                   \
      return RNNT_ERR_CUDA;                            \
    }                                                  \
  } while (0)

// Launch with an optional profiling bracket (see include/rnnt_profile.h).
#define LAUNCH(name, expr)              \
  do {                                  \
    rnnt::ProfScope ps_(name, st);      \
    RNNT_CHECK(expr);                   \
  } while (0)

}  // namespace

rnnt_status rnnt::chunk_count(const Plan& p, const SavedView& sv, cudaStream_t st,
                              long long* n) {
  const long long bound = cdiv(p.max_tiles, p.chunk_tiles);
  if (bound <= 1) {
    *n = bound;
    return RNNT_OK;
  }
  int32_t total = 0;
  RNNT_CHECK(cudaMemcpyAsync(&total, sv.total_tiles, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  RNNT_CHECK(cudaStreamSynchronize(st));
  *n = cdiv(total, p.chunk_tiles);
  return RNNT_OK;
}

ChunkArgs rnnt::chunk_args(const Plan& p, const SavedView& sv, long long k,
                           const int32_t* labels, const int32_t* T_len, const int32_t* U_len) {
  ChunkArgs c;
  c.sh = shape_of(p);
  c.first_tile = k * p.chunk_tiles;
  c.ntiles = p.chunk_tiles;
  c.T_len = T_len;
  c.U_len = U_len;
  c.labels = labels;
  c.sv = sv;
  return c;
}

namespace {

// Projections pA = hA W^A^T + b^Z [B*T,H] and pL = hL W^L^T [B*U1,H], fp32.
rnnt_status projections(const Plan& p, const void* hA, const void* hL, const rnnt_params* pr,
                        float* pA, float* pL, cudaStream_t st, cudaStream_t st_l) {
  const int bf = p.dtype != RNNT_F32;
  if (p.tc) {
    RNNT_CHECK(tc_projection(p, hA, pr->WA, pr->bZ, p.B * p.T, p.HA, pA, st));
    RNNT_CHECK(tc_projection(p, hL, pr->WL, nullptr, p.B * p.U1, p.HL, pL, st_l));
    return RNNT_OK;
  }
  SimtGemm g{};
  g.M = p.B * p.T; g.N = p.H; g.K = p.HA;
  g.A = hA; g.sam = p.HA; g.sak = 1; g.a_bf16 = bf;
  g.Bm = pr->WA; g.sbk = 1; g.sbn = p.HA; g.b_bf16 = bf;
  g.C = pA; g.ldc = p.H; g.alpha = 1.f; g.bias = pr->bZ; g.bias_bf16 = bf;
  LAUNCH("simt_gemm", launch_simt_gemm(g, st));
  g.M = p.B * p.U1; g.K = p.HL;
  g.A = hL; g.sam = p.HL;
  g.Bm = pr->WL; g.sbn = p.HL;
  g.C = pL; g.bias = nullptr;
  LAUNCH("simt_gemm", launch_simt_gemm(g, st));
  return RNNT_OK;
}

// Scores of a chunk on the fp32 path: Hs = Z W^O^T + b^O.
rnnt_status simt_scores(const Plan& p, const rnnt_params* pr, const float* Z, float* Hs,
                        long long rows, cudaStream_t st) {
  const int bf = p.dtype != RNNT_F32;
  SimtGemm g{};
  g.M = (int)rows; g.N = p.V; g.K = p.H;
  g.A = Z; g.sam = p.H; g.sak = 1; g.a_bf16 = 0;
  g.Bm = pr->WO; g.sbk = 1; g.sbn = p.H; g.b_bf16 = bf;
  g.C = Hs; g.ldc = p.V; g.alpha = 1.f; g.bias = pr->bO; g.bias_bf16 = bf;
  LAUNCH("simt_gemm", launch_simt_gemm(g, st));
  return RNNT_OK;
}

rnnt_status check_common(const rnnt_dims* dims, const void* hA, const void* hL,
                         const rnnt_params* pr, const int32_t* labels, const int32_t* T_len,
                         const int32_t* U_len, void* saved, void* ws, size_t ws_bytes,
                         Plan* p) {
  if (!make_plan(dims, p)) return RNNT_ERR_INVALID_ARG;
  if (p->mode == RNNT_UNTILED) {
    // Untiled mode keeps every position's z and scores in `saved`: a plan
    // whose saved state exceeds the device's memory is refused first, before
    // any buffer is looked at (the 40 s, batch-1024 lattice would need ~0.9 TB)
    size_t free_b = 0, total_b = 0;
    if (cudaMemGetInfo(&free_b, &total_b) == cudaSuccess && p->s_total > total_b)
      return RNNT_ERR_WORKSPACE_TOO_SMALL;
  }
  if (!pr || !saved || !ws) return RNNT_ERR_INVALID_ARG;
  if (!aligned(saved) || !aligned(ws)) return RNNT_ERR_INVALID_ARG;
  if (p->B > 0 && (!hA || !hL || !labels || !T_len || !U_len)) return RNNT_ERR_INVALID_ARG;
  if (!pr->WA || !pr->WL || !pr->WO) return RNNT_ERR_INVALID_ARG;
  if (p->U1 > 1024) return RNNT_ERR_UNSUPPORTED_SHAPE;  // one thread per label position
  if (p->T > 65535) return RNNT_ERR_UNSUPPORTED_SHAPE;  // tile table packs T_b in 16 bits
  if (p->tc) {
    // operands of TMA loads and 16-byte vector loads: an unaligned one would
    // fault the kernel, so it is refused here, before any launch
    if (!aligned16(hA) || !aligned16(hL) || !aligned16(pr->WA) || !aligned16(pr->WL) ||
        !aligned16(pr->WO) || !aligned16(pr->bZ) || !aligned16(pr->bO))
      return RNNT_ERR_INVALID_ARG;
    rnnt_status s = tc_check_shape(*p);
    if (s != RNNT_OK) return s;
  }
  if (ws_bytes < p->w_total) return RNNT_ERR_WORKSPACE_TOO_SMALL;
  return RNNT_OK;
}

}  // namespace

extern "C" {

size_t rnnt_saved_bytes(const rnnt_dims* dims) {
  Plan p;
  return make_plan(dims, &p) ? p.s_total : 0;
}

size_t rnnt_workspace_bytes(const rnnt_dims* dims) {
  Plan p;
  return make_plan(dims, &p) ? p.w_total : 0;
}

long long rnnt_tile_cells_for_budget(const rnnt_dims* dims, size_t budget_bytes) {
  if (!dims || dims->mode != RNNT_TILED) return 0;
  rnnt_dims d = *dims;
  Plan p;
  auto footprint = [&](long long tiles) -> size_t {  // 0: invalid
    d.tile_cells = tiles * TILE;
    return make_plan(&d, &p) ? p.s_total + p.w_total : 0;
  };
  d.tile_cells = TILE;
  if (!make_plan(&d, &p)) return 0;
  const long long max_tiles = p.max_tiles;
  if (max_tiles < 1) return 0;
  const size_t one = footprint(1);
  if (one == 0 || one > budget_bytes) return 0;
  if (footprint(max_tiles) <= budget_bytes) return max_tiles * TILE;
  // the footprint grows with the tiles per chunk: largest that fits
  long long lo = 1, hi = max_tiles;  // fits(lo), !fits(hi)
  while (hi - lo > 1) {
    const long long mid = lo + (hi - lo) / 2;
    const size_t f = footprint(mid);
    if (f != 0 && f <= budget_bytes) lo = mid;
    else hi = mid;
  }
  // whole waves of SMs when at least one fits
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      sms > 0 && lo >= sms)
    lo = lo / sms * sms;
  else
    cudaGetLastError();  // (no device: no rounding; clear the error state)
  return lo * TILE;
}

int rnnt_graph_capturable(const rnnt_dims* dims) {
  Plan p;
  if (!make_plan(dims, &p)) return -1;
  return cdiv(p.max_tiles, p.chunk_tiles) <= 1 ? 1 : 0;
}

rnnt_status rnnt_saved_layout(const rnnt_dims* dims, rnnt_saved_offsets* out) {
  Plan p;
  if (!out || !make_plan(dims, &p)) return RNNT_ERR_INVALID_ARG;
  out->status = p.s_status;
  out->lnP = p.s_lnP;
  out->lpb = p.s_lpb;
  out->lpl = p.s_lpl;
  out->lnPD = p.s_lnPD;
  out->alpha = p.s_alpha;
  out->beta = p.s_beta;
  out->z = p.s_z;
  out->h = p.s_h;
  out->total = p.s_total;
  return RNNT_OK;
}

const char* rnnt_status_string(rnnt_status s) {
  switch (s) {
    case RNNT_OK: return "ok";
    case RNNT_ERR_INVALID_ARG: return "invalid argument";
    case RNNT_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case RNNT_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case RNNT_ERR_LENGTH_RANGE: return "length out of range";
    case RNNT_ERR_LABEL_RANGE: return "label out of range";
    case RNNT_ERR_TIMEOUT: return "device wait timed out";
    case RNNT_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

}  // extern "C"

// The forward pass; side_streams = false keeps every launch on `stream`
// (the no-allocation entry point creates no streams).
rnnt_status rnnt::fwd_impl(const rnnt_dims* dims, const void* hA, const void* hL,
                          const rnnt_params* pr, const int32_t* labels, const int32_t* T_len,
                          const int32_t* U_len, float* loss, void* saved, void* ws,
                          size_t ws_bytes, rnnt_stream stream, bool side_streams) {
  Plan p;
  rnnt_status st0 = check_common(dims, hA, hL, pr, labels, T_len, U_len, saved, ws, ws_bytes, &p);
  if (st0 != RNNT_OK) return st0;
  if (p.B > 0 && !loss) return RNNT_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const Shape sh = shape_of(p);
  SavedView sv = saved_view(p, saved);
  char* w = (char*)ws;
  float* pA = (float*)((char*)saved + p.s_pA);
  float* pL = (float*)((char*)saved + p.s_pL);

  rnnt_status s;
  {
    // the two joint projections (they read only the inputs and write only
    // pA, pL) and the -inf fill of the saved arrays run beside the index and
    // tile table
    Fork fork(st, side_streams && p.tc && p.B > 0 ? 3 : 0);
    LAUNCH("index", launch_index(sh, labels, T_len, U_len, sv, loss, st));
    if (p.B == 0) return RNNT_OK;
    s = projections(p, hA, hL, pr, pA, pL, fork.side(0), fork.side(1));
    if (s != RNNT_OK) return s;
    {
      // lpb, lpl, lnPD, alpha, beta are consecutive (with alignment gaps): one fill
      cudaStream_t st = fork.side(2);
      LAUNCH("fill_f32", launch_fill_f32(sv.lpb, -INFINITY,
                                         (p.s_beta - p.s_lpb) / 4 + (size_t)p.B * p.T * p.U1, st));
    }
    LAUNCH("tile_table", launch_tile_table(sh, T_len, U_len, sv, st));
    RNNT_CHECK(fork.join());
  }

  const bool untiled = p.mode == RNNT_UNTILED;
  void* Z = untiled ? (char*)saved + p.s_z : w + p.w_z;
  void* Hs = untiled ? (char*)saved + p.s_h : w + p.w_h;
  if (p.tc) {
    TcF8 f8{};
    if (p.f8) {
      f8 = TcF8{(unsigned char*)(w + p.w_z8), w + p.w_wo8, w + p.w_wodq, (float*)(w + p.w_nscale)};
      LAUNCH("tc_quantize_wo", tc_quantize_wo(p, pr->WO, w + p.w_wo8, w + p.w_wodq,
                                              (float*)(w + p.w_nscale), st));
    }
    s = tc_forward_tiles(p, sv, pr, labels, T_len, U_len, pA, pL, Z, untiled ? Hs : nullptr,
                         p.f8 ? &f8 : nullptr, st);
    if (s != RNNT_OK) return s;
  } else {
    long long nch = 0;
    s = chunk_count(p, sv, st, &nch);
    if (s != RNNT_OK) return s;
    for (long long k = 0; k < nch; ++k) {
      ChunkArgs c = chunk_args(p, sv, k, labels, T_len, U_len);
      LAUNCH("build_z", launch_build_z(c, pA, pL, Z, 0, st));
      s = simt_scores(p, pr, (const float*)Z, (float*)Hs, p.chunk_rows, st);
      if (s != RNNT_OK) return s;
      LAUNCH("lse_rows", launch_lse_rows(c, (const float*)Hs, st));
    }
  }
  LAUNCH("alpha_beta", launch_alpha_beta(sh, T_len, U_len, sv, loss, p.tc, st));
  return RNNT_OK;
}

extern "C" {

rnnt_status rnnt_fwd(const rnnt_dims* dims, const void* hA, const void* hL,
                     const rnnt_params* pr, const int32_t* labels, const int32_t* T_len,
                     const int32_t* U_len, float* loss, void* saved, void* ws, size_t ws_bytes,
                     rnnt_stream stream) {
  return rnnt::fwd_impl(dims, hA, hL, pr, labels, T_len, U_len, loss, saved, ws, ws_bytes,
                        stream, true);
}

rnnt_status rnnt_bwd(const rnnt_dims* dims, const void* hA, const void* hL,
                     const rnnt_params* pr, const int32_t* labels, const int32_t* T_len,
                     const int32_t* U_len, const float* grad_loss, void* saved, float* dhA,
                     float* dhL, float* dWA, float* dWL, float* dbZ, float* dWO, float* dbO,
                     void* ws, size_t ws_bytes, rnnt_stream stream) {
  return rnnt::bwd_impl(dims, hA, hL, pr, labels, T_len, U_len, grad_loss, saved, dhA, dhL, dWA,
                        dWL, dbZ, dWO, dbO, ws, ws_bytes, stream, false);
}

rnnt_status rnnt_bwd_ex(const rnnt_dims* dims, const void* hA, const void* hL,
                        const rnnt_params* pr, const int32_t* labels, const int32_t* T_len,
                        const int32_t* U_len, const float* grad_loss, void* saved, void* dhA,
                        void* dhL, float* dWA, float* dWL, float* dbZ, float* dWO, float* dbO,
                        void* ws, size_t ws_bytes, const rnnt_bwd_opts* opts,
                        rnnt_stream stream) {
  return rnnt::bwd_impl(dims, hA, hL, pr, labels, T_len, U_len, grad_loss, saved, dhA, dhL, dWA,
                        dWL, dbZ, dWO, dbO, ws, ws_bytes, stream, false, opts);
}

rnnt_status rnnt_fwd_bwd(const rnnt_dims* dims, const void* hA, const void* hL,
                         const rnnt_params* pr, const int32_t* labels, const int32_t* T_len,
                         const int32_t* U_len, float* loss, const float* grad_loss, void* saved,
                         float* dhA, float* dhL, float* dWA, float* dWL, float* dbZ, float* dWO,
                         float* dbO, void* ws, size_t ws_bytes, rnnt_stream stream) {
  rnnt_status s = rnnt::fwd_impl(dims, hA, hL, pr, labels, T_len, U_len, loss, saved, ws,
                                 ws_bytes, stream, true);
  if (s != RNNT_OK) return s;
  // the forward's z of a single-chunk plan is still in the workspace
  return rnnt::bwd_impl(dims, hA, hL, pr, labels, T_len, U_len, grad_loss, saved, dhA, dhL, dWA,
                        dWL, dbZ, dWO, dbO, ws, ws_bytes, stream, true);
}

}  // extern "C"

// The backward pass.  z_resident: the workspace still holds the z tiles the
// forward built (rnnt_fwd_bwd), so that a single-chunk plan skips its rebuild.
rnnt_status rnnt::bwd_impl(const rnnt_dims* dims, const void* hA, const void* hL,
                           const rnnt_params* pr, const int32_t* labels, const int32_t* T_len,
                           const int32_t* U_len, const float* grad_loss, void* saved,
                           void* dhA, void* dhL, float* dWA, float* dWL, float* dbZ,
                           float* dWO, float* dbO, void* ws, size_t ws_bytes,
                           rnnt_stream stream, bool z_resident, const rnnt_bwd_opts* opts) {
  Plan p;
  rnnt_status st0 = check_common(dims, hA, hL, pr, labels, T_len, U_len, saved, ws, ws_bytes, &p);
  if (st0 != RNNT_OK) return st0;
  EncOut eout{false, nullptr, nullptr};
  if (opts) {
    if (opts->enc_grad_dtype != RNNT_F32 && opts->enc_grad_dtype != RNNT_BF16)
      return RNNT_ERR_INVALID_ARG;
    eout = EncOut{opts->enc_grad_dtype == RNNT_BF16, opts->dA, opts->dL};
    if (eout.bf16 && !p.tc) return RNNT_ERR_INVALID_ARG;  // bf16 hand-off: bf16 problems
  }
  // the tensor-core path writes these by 16-byte stores and vector reductions
  // (and reads a bf16 dA / dL back by TMA)
  if (p.tc) {
    const void* outs[7] = {dhA, dhL, dWA, dWL, dWO, eout.dA, eout.dL};
    for (const void* o : outs)
      if (!aligned16(o)) return RNNT_ERR_INVALID_ARG;
  }
  cudaStream_t st = (cudaStream_t)stream;
  SavedView sv = saved_view(p, saved);
  char* w = (char*)ws;
  const float* pA = (const float*)((char*)saved + p.s_pA);  // written by rnnt_fwd
  const float* pL = (const float*)((char*)saved + p.s_pL);
  float* dA = (float*)(w + p.w_dA);
  float* dLr = (float*)(w + p.w_dLr);
  int32_t* Teff = (int32_t*)(w + p.w_len);
  int32_t* Ueff = Teff + (p.B ? p.B : 1);
  const int bf = p.dtype != RNNT_F32;
  const bool untiled = p.mode == RNNT_UNTILED;

  // Outputs are overwritten; accumulated ones start from zero (one launch).
  if (p.B == 0) {
    ZeroList z0{};
    void* ps0[5] = {dWO, dbO, dbZ, dWA, dWL};
    size_t bs0[5] = {sizeof(float) * (size_t)p.V * p.H, sizeof(float) * (size_t)p.V,
                     sizeof(float) * (size_t)p.H, sizeof(float) * (size_t)p.H * p.HA,
                     sizeof(float) * (size_t)p.H * p.HL};
    for (int i = 0; i < 5; ++i) { z0.p[z0.n] = ps0[i]; z0.bytes[z0.n] = bs0[i]; ++z0.n; }
    LAUNCH("zero", launch_zero_many(z0, st));
    return RNNT_OK;
  }
  // tensor-core path: db^O is summed into an aligned workspace vector and
  // copied to the caller's (any alignment) at the end
  float* dbO_acc = (p.tc && dbO) ? (float*)(w + p.w_dbO) : dbO;
  // zero the accumulated outputs (one launch) and clamp the lengths
  auto prepare = [&](cudaStream_t st) -> rnnt_status {
    ZeroList z{};
    void* ps[7] = {dWO, dbO_acc, dbZ, dA, dLr, dWA, dWL};
    size_t bs[7] = {sizeof(float) * (size_t)p.V * p.H, sizeof(float) * (size_t)p.V,
                    sizeof(float) * (size_t)p.H, sizeof(float) * (size_t)p.B * p.T * p.H,
                    sizeof(float) * (size_t)p.B * p.U1 * p.H, sizeof(float) * (size_t)p.H * p.HA,
                    sizeof(float) * (size_t)p.H * p.HL};
    for (int i = 0; i < 7; ++i) { z.p[z.n] = ps[i]; z.bytes[z.n] = bs[i]; ++z.n; }
    LAUNCH("zero", launch_zero_many(z, st));
    LAUNCH("eff_lengths", launch_eff_lengths(shape_of(p), sv, T_len, U_len, Teff, Ueff, st));
    return RNNT_OK;
  };

  rnnt_status s;
  void* Z = untiled ? (char*)saved + p.s_z : w + p.w_z;
  void* Hs = untiled ? (char*)saved + p.s_h : w + p.w_h;

  if (p.tc) {
    TcF8 f8{};
    if (p.f8) {
      f8 = TcF8{(unsigned char*)(w + p.w_z8), w + p.w_wo8, w + p.w_wodq, (float*)(w + p.w_nscale)};
      LAUNCH("tc_quantize_wo", tc_quantize_wo(p, pr->WO, w + p.w_wo8, w + p.w_wodq,
                                              (float*)(w + p.w_nscale), st));
    }
    // (the preparation runs beside the first chunk's z rebuild, the
    // encoder-side gradients beside the last chunk's dW^O)
    const PreLaunch pre = prepare;
    const PreLaunch enc = [&](cudaStream_t es) {
      return tc_encoder_grads(p, w, hA, hL, pr, Teff, Ueff, dA, dLr, dhA, dhL, dWA, dWL, dbZ,
                              eout, es);
    };
    s = tc_backward_tiles(p, sv, pr, labels, T_len, U_len, grad_loss, pA, pL, Z, Hs, untiled,
                          z_resident, dA, dLr, dWO, dbO_acc, (float4*)(w + p.w_post),
                          p.f8 ? &f8 : nullptr, &pre, &enc, st);
    if (s != RNNT_OK) return s;
    if (dbO)
      RNNT_CHECK(cudaMemcpyAsync(dbO, dbO_acc, sizeof(float) * (size_t)p.V,
                                 cudaMemcpyDeviceToDevice, st));
    return RNNT_OK;
  }

  s = prepare(st);
  if (s != RNNT_OK) return s;
  long long nch = 0;
  s = chunk_count(p, sv, st, &nch);
  if (s != RNNT_OK) return s;
  float* dZ = (float*)(w + p.w_dz);
  for (long long k = 0; k < nch; ++k) {
    ChunkArgs c = chunk_args(p, sv, k, labels, T_len, U_len);
    if (!untiled) {
      LAUNCH("build_z", launch_build_z(c, pA, pL, Z, 0, st));
      s = simt_scores(p, pr, (const float*)Z, (float*)Hs, p.chunk_rows, st);
      if (s != RNNT_OK) return s;
    }
    LAUNCH("dh_rows", launch_dh_rows(c, (float*)Hs, grad_loss, st));
    // dz = dh W^O
    SimtGemm g{};
    g.M = (int)p.chunk_rows; g.N = p.H; g.K = p.V;
    g.A = Hs; g.sam = p.V; g.sak = 1;
    g.Bm = pr->WO; g.sbk = p.H; g.sbn = 1; g.b_bf16 = bf;
    g.C = dZ; g.ldc = p.H; g.alpha = 1.f;
    LAUNCH("simt_gemm", launch_simt_gemm(g, st));
    LAUNCH("da_reduce", launch_da_reduce(c, dZ, Z, 0, dA, dLr, st));
    if (dWO) {  // dW^O += dh^T z
      SimtGemm q{};
      q.M = p.V; q.N = p.H; q.K = (int)p.chunk_rows;
      q.A = Hs; q.sam = 1; q.sak = p.V;
      q.Bm = Z; q.sbk = p.H; q.sbn = 1;
      q.C = dWO; q.ldc = p.H; q.alpha = 1.f; q.accumulate = 1;
      LAUNCH("simt_gemm", launch_simt_gemm(q, st));
    }
    if (dbO) LAUNCH("colsum", launch_colsum((const float*)Hs, p.chunk_rows, p.V, p.V, dbO, st));
  }

  // Encoder-side gradients from the reduced pre-activation gradients.
  SimtGemm g{};
  if (dhA) {  // dh^A = dA W^A
    g = SimtGemm{};
    g.M = p.B * p.T; g.N = p.HA; g.K = p.H;
    g.A = dA; g.sam = p.H; g.sak = 1;
    g.Bm = pr->WA; g.sbk = p.HA; g.sbn = 1; g.b_bf16 = bf;
    g.C = (float*)dhA; g.ldc = p.HA; g.alpha = 1.f;
    LAUNCH("simt_gemm", launch_simt_gemm(g, st));
  }
  if (dWA) {  // dW^A = dA^T hA over the frames of accepted samples
    g = SimtGemm{};
    g.M = p.H; g.N = p.HA; g.K = p.B * p.T;
    g.A = dA; g.sam = 1; g.sak = p.H;
    g.Bm = hA; g.sbk = p.HA; g.sbn = 1; g.b_bf16 = bf;
    g.C = dWA; g.ldc = p.HA; g.alpha = 1.f;
    g.kmask_len = Teff; g.kperiod = p.T; g.kmask_off = 0;
    LAUNCH("simt_gemm", launch_simt_gemm(g, st));
  }
  if (dhL) {
    g = SimtGemm{};
    g.M = p.B * p.U1; g.N = p.HL; g.K = p.H;
    g.A = dLr; g.sam = p.H; g.sak = 1;
    g.Bm = pr->WL; g.sbk = p.HL; g.sbn = 1; g.b_bf16 = bf;
    g.C = (float*)dhL; g.ldc = p.HL; g.alpha = 1.f;
    LAUNCH("simt_gemm", launch_simt_gemm(g, st));
  }
  if (dWL) {
    g = SimtGemm{};
    g.M = p.H; g.N = p.HL; g.K = p.B * p.U1;
    g.A = dLr; g.sam = 1; g.sak = p.H;
    g.Bm = hL; g.sbk = p.HL; g.sbn = 1; g.b_bf16 = bf;
    g.C = dWL; g.ldc = p.HL; g.alpha = 1.f;
    g.kmask_len = Ueff; g.kperiod = p.U1; g.kmask_off = 0;
    LAUNCH("simt_gemm", launch_simt_gemm(g, st));
  }
  if (dbZ) LAUNCH("colsum", launch_colsum(dA, (long long)p.B * p.T, p.H, p.H, dbZ, st));
  // the projections' gradients handed over (fp32 on this path)
  if (eout.dA)
    RNNT_CHECK(cudaMemcpyAsync(eout.dA, dA, sizeof(float) * (size_t)p.B * p.T * p.H,
                               cudaMemcpyDeviceToDevice, st));
  if (eout.dL)
    RNNT_CHECK(cudaMemcpyAsync(eout.dL, dLr, sizeof(float) * (size_t)p.B * p.U1 * p.H,
                               cudaMemcpyDeviceToDevice, st));
  return RNNT_OK;
}

extern "C" {

rnnt_status rnnt_device_status(const rnnt_dims* dims, const void* saved, rnnt_stream stream,
                               int32_t* word) {
  Plan p;
  if (!make_plan(dims, &p) || !saved) return RNNT_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t w = 0;
  RNNT_CHECK(cudaMemcpyAsync(&w, (const char*)saved + p.s_status, sizeof(int32_t),
                             cudaMemcpyDeviceToHost, st));
  RNNT_CHECK(cudaStreamSynchronize(st));
  if (word) *word = w;
  const rnnt_status order[] = {RNNT_ERR_LENGTH_RANGE, RNNT_ERR_LABEL_RANGE, RNNT_ERR_TIMEOUT};
  for (rnnt_status c : order)
    if (w & status_bit(c)) return c;
  return RNNT_OK;
}

}  // extern "C"
