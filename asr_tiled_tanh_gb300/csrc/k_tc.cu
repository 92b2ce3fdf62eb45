// k_tc.cu -- bf16 tensor-core path (placeholder until the tcgen05 kernels land).
#include "tc.h"

namespace rnnt {

bool tc_path_enabled() { return false; }
rnnt_status tc_check_shape(const Plan&) { return RNNT_ERR_UNSUPPORTED_SHAPE; }
cudaError_t tc_projection(const Plan&, const void*, const void*, const void*, int, int, float*,
                          cudaStream_t) {
  return cudaErrorNotSupported;
}
rnnt_status tc_forward_tiles(const Plan&, const SavedView&, const rnnt_params*, const int32_t*,
                             const int32_t*, const int32_t*, const float*, const float*, void*,
                             void*, cudaStream_t) {
  return RNNT_ERR_UNSUPPORTED_SHAPE;
}
rnnt_status tc_backward_tiles(const Plan&, const SavedView&, const rnnt_params*, const int32_t*,
                              const int32_t*, const int32_t*, const float*, const float*,
                              const float*, void*, void*, bool, float*, float*, float*, float*,
                              cudaStream_t) {
  return RNNT_ERR_UNSUPPORTED_SHAPE;
}
rnnt_status tc_encoder_grads(const Plan&, char*, const void*, const void*, const rnnt_params*,
                             const int32_t*, const int32_t*, float*, float*, float*, float*,
                             float*, float*, float*, cudaStream_t) {
  return RNNT_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace rnnt
