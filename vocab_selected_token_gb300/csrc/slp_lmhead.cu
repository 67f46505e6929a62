// Fused LM-head path (not built yet).
#include "slp_internal.h"

namespace slp {

size_t lmhead_workspace_size(int64_t, int64_t, int64_t) { return 256; }

cudaError_t launch_lmhead_forward(const void*, const void*, int64_t, int64_t, int64_t,
                                  const int32_t*, const uint8_t*, float, float*, float*, void*,
                                  int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t launch_lmhead_backward(const void*, const void*, int64_t, int64_t, int64_t,
                                   const int32_t*, const uint8_t*, float, const float*,
                                   const float*, void*, void*, void*, int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace slp
