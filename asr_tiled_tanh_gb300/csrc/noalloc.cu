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
// device address is looked up once per device (cudaGetSymbolAddress, with
// that device current) on the first call made on it, and that address is what
// the kernels receive.
#include <mutex>

#include "../../include/rnnt.h"
#include "kernels.h"
#include <cuda_runtime.h>

namespace {

constexpr size_t kScratchBytes = (size_t)RNNT_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_setup_mu;

// Device address of g_scratch on the current device (set up on first use).
rnnt_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RNNT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return RNNT_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
  rnnt_status s = scratch_on_current_device(&ws);
  if (s != RNNT_OK) return s;
  // The forward overwrites every scratch byte it reads, so nothing left over
  // from an earlier call has to be cleared first.
  // (all on `stream`: the plain forward's side streams are not created here)
  return rnnt::fwd_impl(dims, hA, hL, params, labels, T_len, U_len, loss, saved, ws,
                        kScratchBytes, stream, false);
}
