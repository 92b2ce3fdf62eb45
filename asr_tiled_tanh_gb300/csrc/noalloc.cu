// noalloc.cu -- rnnt_fwd_noalloc: the forward pass with its scratch memory in a
// fixed, file-scope device array, for callers that cannot allocate.
//
// Who needs this: hosts that reserve all device memory up front and forbid
// cudaMalloc afterwards (fixed-pool runtimes), plugin interfaces that hand the
// callee inputs and outputs but no allocator, and latency-critical loops
// where an allocation, or its failure, is not acceptable.  Such a caller can
// still provide `saved` and `loss` (outputs), but not the scratch buffer `ws`
// that rnnt_fwd asks for.
//
// How: the scratch lives in g_scratch below, RNNT_NOALLOC_SCRATCH_BYTES bytes
// that every GPU loading this library reserves until the process exits.  In
// host code `g_scratch` names a host-side stand-in, not device memory, so the
// device address is looked up (cudaGetSymbolAddress) the first time a call is
// made in a CUDA context, with that context current, and that address is what
// the kernels receive.  The address belongs to the context, not to the device
// ordinal: a host that drives the GPU through its own (non-primary) context,
// or that reset the device (a new primary context), gets the address of the
// array in the context that is current at the call.  Contexts are told apart
// by their unique ID (cuCtxGetId), which a context created after a reset never
// shares with the one before it.
#include <cuda.h>

#include <mutex>

#include "../../include/rnnt.h"
#include "kernels.h"
#include <cuda_runtime.h>

namespace {

constexpr size_t kScratchBytes = (size_t)RNNT_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Address of g_scratch per context, keyed by the context's unique ID.
constexpr int kMaxContexts = 64;
struct ScratchSlot {
  unsigned long long ctx_id;
  void* ptr;
};
ScratchSlot g_slots[kMaxContexts] = {};
int g_nslots = 0;
std::mutex g_setup_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Driver entry points for the current context and its ID (null when the
// driver does not provide them).
void driver_fns(CtxGetCurrentFn* cur, CtxGetIdFn* id) {
  static CtxGetCurrentFn f_cur = nullptr;
  static CtxGetIdFn f_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f_cur = (CtxGetCurrentFn)f;
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f_id = (CtxGetIdFn)f;
  });
  *cur = f_cur;
  *id = f_id;
}

// Unique ID of the current context, or false when there is none yet (the
// runtime creates the primary context on its first use) or the driver has no
// context IDs.
bool current_context_id(unsigned long long* id) {
  CtxGetCurrentFn f_cur;
  CtxGetIdFn f_id;
  driver_fns(&f_cur, &f_id);
  CUcontext ctx = nullptr;
  return f_cur && f_id && f_cur(&ctx) == CUDA_SUCCESS && ctx && f_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch in the current context (looked up on the first
// call made in that context).
rnnt_status scratch_in_current_context(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return RNNT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  unsigned long long id = 0;
  if (current_context_id(&id)) {
    for (int i = 0; i < g_nslots; ++i)
      if (g_slots[i].ctx_id == id) {
        *out = g_slots[i].ptr;
        return RNNT_OK;
      }
  }
  // (the lookup makes the device's primary context current if no context was)
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return RNNT_ERR_CUDA;
  // without a context ID the lookup is repeated on every call (it allocates nothing)
  if (current_context_id(&id)) {
    const int i = g_nslots < kMaxContexts ? g_nslots++ : (int)(id % kMaxContexts);
    g_slots[i] = ScratchSlot{id, p};
  }
  *out = p;
  return RNNT_OK;
}

}  // namespace

extern "C" rnnt_status rnnt_fwd_noalloc(const rnnt_dims* dims, const void* hA, const void* hL,
                                        const rnnt_params* params, const int32_t* labels,
                                        const int32_t* T_len, const int32_t* U_len, float* loss,
                                        void* saved, rnnt_stream stream) {
  const size_t need = rnnt_workspace_bytes(dims);
  if (need == 0) return RNNT_ERR_INVALID_ARG;
  if (need > kScratchBytes) return RNNT_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  rnnt_status s = scratch_in_current_context(&ws);
  if (s != RNNT_OK) return s;
  // The forward overwrites every scratch byte it reads, so nothing left over
  // from an earlier call has to be cleared first.
  // (all on `stream`: the plain forward's side streams are not created here)
  return rnnt::fwd_impl(dims, hA, hL, params, labels, T_len, U_len, loss, saved, ws,
                        kScratchBytes, stream, false);
}
