/*
 * rnnt.h -- C ABI of the GB300 (sm_103a) RNN-T joint network + output layer +
 * transducer loss library (librnnt_gb300.so).
 *
 * The operation is the one stated in "Neural transducer training: reduced
 * memory consumption with sample-wise computation" (arXiv 2211.16270), §2:
 *   joint network  (Eq. 3-4)  z[b,t,u] = tanh(W^A hA[b,t] + W^L hL[b,u] + b^Z)
 *   output layer   (Eq. 5-6)  h[b,t,u] = W^O z[b,t,u] + b^O
 *   loss f^W_1..4  (Eq. 7-10) softmax denominator P_D, forward/backward
 *                             variables alpha/beta, L = -sum_b ln P(y_b|x_b),
 *                             and dh = dL/dh,
 * followed by the backward pass through the output layer and joint network
 * (§4, Algorithm 1: dtheta^J, dtheta^O and the encodings' gradients).  The
 * execution follows the tiled scheme of the Flash RNN-T blog ("Compute it, use
 * it, make room"): the forward keeps only the blank and label log-probabilities
 * of each lattice position, the backward recomputes each tile of positions and
 * overwrites its scores with their gradients ("Making each operation more
 * efficient").  RNNT_UNTILED keeps the joint intermediates instead.
 *
 * Conventions (all calls):
 *  - All tensor pointers are DEVICE pointers, row-major and contiguous, except
 *    the rnnt_dims / rnnt_params structs themselves, which are host memory.
 *  - labels[b,0] is the prepended blank (§2) and is never read; the move from
 *    label position u to u+1 emits labels[b,u+1].  hL row u is the label
 *    context after u labels.  Lattice of sample b: t < T_len[b],
 *    u <= U_len[b].  Rows of hA/hL and labels beyond a sample's lengths are
 *    never read (they may hold anything, NaN included).
 *  - The caller owns every buffer.  The library never allocates device
 *    memory; it uses the `saved` and `ws` buffers it is given.
 *  - Every call is asynchronous on `stream`, except where noted.  Calls that
 *    share a `ws` or `saved` buffer must not run concurrently.
 *  - Host-checkable problems (NULL pointers, bad dims, unsupported shapes,
 *    buffers too small) return an error before anything is launched.
 *    Problems only the device can see (lengths out of range, labels out of
 *    range) set bits in the device status word kept in `saved`; the affected
 *    sample gets loss NaN and contributes nothing to any gradient.  Read the
 *    word with rnnt_device_status.  No kernel traps or asserts.
 */
#ifndef RNNT_GB300_H
#define RNNT_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque stand-in for cudaStream_t (same representation: a pointer). */
typedef void* rnnt_stream;

typedef enum {
  RNNT_OK = 0,
  RNNT_ERR_INVALID_ARG = 1,        /* NULL pointer, negative or zero size, bad enum */
  RNNT_ERR_UNSUPPORTED_SHAPE = 2,  /* shape this build's kernels do not handle */
  RNNT_ERR_WORKSPACE_TOO_SMALL = 3,/* ws_bytes < rnnt_workspace_bytes(), or an
                                      untiled plan whose saved state exceeds the
                                      device's memory (checked first, before any
                                      pointer argument) */
  RNNT_ERR_LENGTH_RANGE = 4,       /* device: some T_len not in [1,T] or U_len not in [0,U1-1] */
  RNNT_ERR_LABEL_RANGE = 5,        /* device: some labels[b,1..U_len[b]] not in [0,V) */
  RNNT_ERR_TIMEOUT = 6,            /* device: a bounded wait inside a kernel gave up */
  RNNT_ERR_CUDA = 7                /* a CUDA runtime call failed (launch, copy, ...) */
} rnnt_status;

typedef enum { RNNT_F32 = 0, RNNT_BF16 = 1, RNNT_BF16_E4M3 = 2 } rnnt_dtype;
typedef enum { RNNT_TILED = 0, RNNT_UNTILED = 1 } rnnt_mode;

/* Problem description (host struct).
 *   B, T, U1 (= U+1, label positions including the prepended blank), HA, HL
 *   (encoding sizes), H (joint size), V (vocabulary), blank (blank id in [0,V)).
 *   dtype: element type of hA, hL and every parameter (RNNT_F32 or RNNT_BF16).
 *     RNNT_F32 runs fp32 FFMA kernels end to end; RNNT_BF16 runs the bf16
 *     tensor-core path (tcgen05, fp32 accumulation).
 *     RNNT_BF16_E4M3: bf16 inputs and parameters as RNNT_BF16, with the
 *     output layer's score products (the forward scores and the backward's
 *     recompute, 2 of the 3 H x V products per position) on e4m3 tensor
 *     cores (tcgen05.mma kind::f8f6f4, fp32 accumulation) - the reduced-
 *     precision output layer the sample-wise paper names as complementary
 *     work (§1 Introduction, ref. [11]; §5 Conclusion).  W^O is quantized per
 *     block of 256 rows: S = the smallest power of two with
 *     max|W^O[block]| / S <= 448, q = e4m3(W^O / S) rounded to nearest even,
 *     and the layer computed is W^O_q = q S (exact in bf16) in the forward
 *     and in every backward product; dWO and dbO are the gradients with
 *     respect to W^O_q and b^O (the caller applies them to W^O: the
 *     straight-through reading).  z enters the score products as
 *     e4m3(2^8 z).  Requires H % 16 == 0.
 *   mode: RNNT_TILED (recompute per tile in the backward; workspace set by
 *     tile_cells) or RNNT_UNTILED (z and the scores are kept in `saved` for
 *     every lattice position; no recompute).
 *   tile_cells: lattice positions whose intermediates the backward holds at
 *     once in tiled mode (the Flash RNN-T "tile"); rounded up to a multiple of
 *     128.  0 selects a default.  Ignored in untiled mode. */
typedef struct {
  int B, T, U1, HA, HL, H, V, blank;
  int dtype;
  int mode;
  long long tile_cells;
} rnnt_dims;

/* Parameters theta^J = {W^A [H,HA], W^L [H,HL], b^Z [H]} (§2, joint network)
 * and theta^O = {W^O [V,H], b^O [V]} (§2, output layer); device pointers of
 * dims.dtype.  bZ and bO may be NULL (zero bias). */
typedef struct {
  const void* WA;
  const void* WL;
  const void* bZ;
  const void* WO;
  const void* bO;
} rnnt_params;

/* Byte offsets of the arrays inside `saved` (see rnnt_saved_layout).
 * lpb, lpl, lnPD, alpha, beta: fp32 [B,T,U1], natural-log values:
 *   lnPD = ln sum_v exp h_v (the softmax denominator of Eq. 7), lpb =
 *   h_blank - lnPD, lpl = h_{labels[b,u+1]} - lnPD (-inf on row u = U_len[b]),
 *   alpha/beta the forward/backward variables of Eq. 8.  Every position
 *   outside a sample's lattice holds -inf.
 * lnP: fp32 [B], ln P(y_b|x_b) (NaN for a rejected sample).
 * status: one int32, the device status word: bit k is set when a problem with
 *   rnnt_status code k was detected (see rnnt_device_status).
 * z, h: untiled mode only (otherwise 0): z [cells,H] and the scores / their
 *   gradients [cells,V], element type = dims.dtype, rows in the library's
 *   tile order (not [B,T,U1]). */
typedef struct {
  size_t status, lnP, lpb, lpl, lnPD, alpha, beta, z, h, total;
} rnnt_saved_offsets;

/* Bytes of the `saved` buffer that rnnt_fwd fills and rnnt_bwd reads:
 * 20 B per lattice position [B,T,U1], the joint projections W^A hA + b^Z
 * [B,T,H] and W^L hL [B,U1,H] in fp32 (kept so that the backward rebuilds z
 * without redoing them), small headers, and in untiled mode the kept z and
 * scores.  Returns 0 if dims are invalid. */
size_t rnnt_saved_bytes(const rnnt_dims* dims);

/* Fill *out with the layout of `saved` for dims.  Returns RNNT_OK or
 * RNNT_ERR_INVALID_ARG. */
rnnt_status rnnt_saved_layout(const rnnt_dims* dims, rnnt_saved_offsets* out);

/* Bytes of the scratch buffer `ws` that rnnt_fwd and rnnt_bwd need: the tile
 * buffers (tile_cells x (H + V) elements in tiled mode), the fp32 gradient
 * accumulators of the joint pre-activations [B,T,H] and [B,U1,H], and their
 * bf16 copies for the encoder-side products.  Returns 0 if dims are invalid.
 * The buffer needs no initialisation (its contents are not carried from
 * rnnt_fwd to rnnt_bwd) and 256-byte alignment. */
size_t rnnt_workspace_bytes(const rnnt_dims* dims);

/* Memory-bounded scheduling: the tile_cells for which the library's whole
 * device footprint, rnnt_saved_bytes + rnnt_workspace_bytes, fits in
 * budget_bytes (tiled mode; dims->tile_cells is ignored).  The lattice is
 * walked sample by sample in chunks of tiles (consecutive samples' tiles,
 * padding-free), so the budget bounds how much of the batch is in flight at
 * once while the per-position saved state (20 bytes) and the per-frame
 * vectors stay whole: the Flash RNN-T blog's "Compute it, use it, make room"
 * tile, and the sample-wise paper's conclusion that memory need barely grow
 * with the batch, turned into a size the caller asks for.  Returns the
 * largest multiple of 128 lattice positions that fits, rounded down to whole
 * waves of the current device's SMs when at least one wave fits, capped at
 * the whole lattice (one chunk: no host synchronization, see
 * rnnt_graph_capturable); 0 if not even one tile fits or dims are invalid or
 * untiled. */
long long rnnt_tile_cells_for_budget(const rnnt_dims* dims, size_t budget_bytes);

/* Whether rnnt_fwd and rnnt_bwd for dims run entirely as stream work, with
 * no host-side synchronization, so that a caller can capture them into a
 * CUDA graph: true when every possible lattice tile fits one chunk of the
 * tile buffers (tiled mode with the default or a large enough tile_cells,
 * and untiled mode); otherwise each call reads the actual tile count back to
 * the host once.  The side streams the library forks from `stream` are
 * joined back before each call returns, which capture supports.  Returns 1,
 * 0, or -1 if dims are invalid.  (Not a method step: the pages have no
 * counterpart.) */
int rnnt_graph_capturable(const rnnt_dims* dims);

/* Forward pass.  Inputs: hA [B,T,HA], hL [B,U1,HL], params, labels [B,U1]
 * int32, T_len [B], U_len [B] int32.  Outputs: loss [B] fp32 = -ln P(y_b|x_b)
 * (the batch loss of Eq. 9 is their sum), and `saved` (rnnt_saved_bytes,
 * 256-byte aligned) for rnnt_bwd.  ws: rnnt_workspace_bytes bytes.
 * stream: a cudaStream_t (NULL = legacy default stream).
 * bf16 problems (RNNT_BF16, RNNT_BF16_E4M3: the tensor-core path, which reads
 * its operands by TMA and 16-byte vector loads) need hA, hL and every params
 * array 16-byte aligned; an unaligned one is refused with
 * RNNT_ERR_INVALID_ARG before anything is launched.  The fp32 path has no
 * alignment rule beyond the element size. */
rnnt_status rnnt_fwd(const rnnt_dims* dims, const void* hA, const void* hL,
                     const rnnt_params* params, const int32_t* labels, const int32_t* T_len,
                     const int32_t* U_len, float* loss, void* saved, void* ws, size_t ws_bytes,
                     rnnt_stream stream);

/* Backward pass for sum_b grad_loss[b] * loss[b] (grad_loss NULL = all ones).
 * Takes the same inputs as the matching rnnt_fwd and the `saved` buffer it
 * filled (untiled mode: the kept scores in `saved` are overwritten with their
 * gradients, so a second rnnt_bwd on the same `saved` is not allowed).
 * Outputs, all fp32 and OVERWRITTEN (not accumulated): dhA [B,T,HA],
 * dhL [B,U1,HL], dWA [H,HA], dWL [H,HL], dbZ [H], dWO [V,H], dbO [V].  Rows
 * beyond a sample's lengths are written as 0.  Any output pointer may be NULL
 * to skip writing it (the work that feeds other outputs still runs).
 * When the largest lattice the dims allow does not fit in one tile buffer,
 * this call synchronizes `stream` once to read the number of tiles.
 * bf16 problems: as for rnnt_fwd, and dhA, dhL, dWA, dWL, dWO 16-byte aligned
 * (written by 16-byte stores and vector reductions; dbZ and dbO have no
 * alignment rule), else RNNT_ERR_INVALID_ARG before anything is launched. */
rnnt_status rnnt_bwd(const rnnt_dims* dims, const void* hA, const void* hL,
                     const rnnt_params* params, const int32_t* labels, const int32_t* T_len,
                     const int32_t* U_len, const float* grad_loss, void* saved, float* dhA,
                     float* dhL, float* dWA, float* dWL, float* dbZ, float* dWO, float* dbO,
                     void* ws, size_t ws_bytes, rnnt_stream stream);

/* Options of rnnt_bwd_ex: how the encoder-side gradients are handed over.
 * All zero / NULL gives exactly rnnt_bwd.
 *   enc_grad_dtype: element type of the dhA and dhL outputs, RNNT_F32 (as
 *     rnnt_bwd) or RNNT_BF16 (bf16 [B,T,HA] / [B,U1,HL], round to nearest
 *     even from the fp32 accumulators; half the bytes for an encoder whose
 *     backward runs in bf16).  RNNT_BF16 needs a bf16 problem (dims.dtype
 *     RNNT_BF16 or RNNT_BF16_E4M3).
 *   dA, dL: optional outputs [B,T,H] and [B,U1,H] of element type
 *     enc_grad_dtype: the gradients with respect to the joint network's
 *     projections, dA[b,t] = dL/d(W^A hA[b,t] + b^Z) and
 *     dL[b,u] = dL/d(W^L hL[b,u]) (the pre-activation gradients summed over
 *     the other lattice axis; 0 outside a sample's lengths), so that
 *     dh^A = dA W^A and dh^L = dL W^L.  An encoder can fold these products into
 *     its own first backward GEMM (function merging across the boundary, as
 *     the sample-wise paper's §1 Introduction describes for the loss and
 *     output layer) and pass dhA = dhL = NULL, which skips them here.
 * Not a step of the pages' method: an interface for the caller's backward. */
typedef struct {
  int enc_grad_dtype;
  void* dA;
  void* dL;
} rnnt_bwd_opts;

/* rnnt_bwd with options (opts NULL: rnnt_bwd).  dhA and dhL point to
 * opts->enc_grad_dtype elements (cast through void*).  Extra errors:
 * RNNT_ERR_INVALID_ARG for an unknown enc_grad_dtype, RNNT_BF16 on an fp32
 * problem, or (bf16 problems) an opts->dA / opts->dL that is not 16-byte
 * aligned. */
rnnt_status rnnt_bwd_ex(const rnnt_dims* dims, const void* hA, const void* hL,
                        const rnnt_params* params, const int32_t* labels, const int32_t* T_len,
                        const int32_t* U_len, const float* grad_loss, void* saved, void* dhA,
                        void* dhL, float* dWA, float* dWL, float* dbZ, float* dWO, float* dbO,
                        void* ws, size_t ws_bytes, const rnnt_bwd_opts* opts,
                        rnnt_stream stream);

/* One training step: rnnt_fwd followed by rnnt_bwd on the same buffers, with
 * the arguments of both (loss is written as by rnnt_fwd; grad_loss and the
 * gradient outputs are as for rnnt_bwd) and the same results.  Because the
 * workspace is not handed back to the caller between the two passes, a plan
 * whose lattice fits one chunk (rnnt_graph_capturable) reuses the z tiles
 * that the forward built instead of rebuilding them in the backward; the
 * scores are still recomputed per tile (Flash RNN-T blog, "Compute it, use
 * it, make room").  Errors: those of rnnt_fwd, then those of rnnt_bwd; the
 * backward does not run when the forward returns an error. */
rnnt_status rnnt_fwd_bwd(const rnnt_dims* dims, const void* hA, const void* hL,
                         const rnnt_params* params, const int32_t* labels, const int32_t* T_len,
                         const int32_t* U_len, float* loss, const float* grad_loss,
                         void* saved, float* dhA, float* dhL, float* dWA, float* dWL,
                         float* dbZ, float* dWO, float* dbO, void* ws, size_t ws_bytes,
                         rnnt_stream stream);

/* Size of the fixed device scratch array used by rnnt_fwd_noalloc. */
#define RNNT_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Forward pass for callers that cannot allocate device memory at all: hosts
 * that reserve every byte up front and forbid cudaMalloc afterwards, plugin
 * interfaces that pass inputs and outputs but no allocator, and latency-
 * critical loops where an allocation (or its failure) is not acceptable.
 * The pages have no counterpart; it is a deployment convenience.
 * Same arguments and results as rnnt_fwd, minus `ws`/`ws_bytes`: the scratch
 * comes from one static device array of RNNT_NOALLOC_SCRATCH_BYTES (32 MiB)
 * that every GPU loading this library holds until the process exits.
 * Returns RNNT_ERR_WORKSPACE_TOO_SMALL, before doing anything else, when
 * rnnt_workspace_bytes(dims) exceeds that size (use a smaller tile_cells, or
 * rnnt_fwd with your own buffer).  The first call made in a CUDA context
 * looks up the array's device address in that context (cudaGetSymbolAddress,
 * with the context current): the primary context of the current device, or
 * the caller's own context if one is current; after a device reset the new
 * context gets its own lookup.  Make that first call before any stream
 * capture.  Every
 * call on a device shares the one array and it keeps the last call's
 * contents; the forward needs none of it cleared.  Calls whose work overlaps
 * on the GPU (other streams, other host threads) race on the array and must
 * be serialized by the caller.  Allocates nothing. */
rnnt_status rnnt_fwd_noalloc(const rnnt_dims* dims, const void* hA, const void* hL,
                             const rnnt_params* params, const int32_t* labels,
                             const int32_t* T_len, const int32_t* U_len, float* loss,
                             void* saved, rnnt_stream stream);

/* Synchronize `stream` and read the device status word in `saved`.  Returns
 * RNNT_OK if no device-side problem was recorded, else the first recorded
 * code among RNNT_ERR_LENGTH_RANGE, RNNT_ERR_LABEL_RANGE, RNNT_ERR_TIMEOUT.
 * If `word` is not NULL it receives the raw bitmask (bit k <=> status code k). */
rnnt_status rnnt_device_status(const rnnt_dims* dims, const void* saved, rnnt_stream stream,
                               int32_t* word);

/* Static, human-readable name of a status code. */
const char* rnnt_status_string(rnnt_status s);

#ifdef __cplusplus
}
#endif
#endif /* RNNT_GB300_H */
