// slp_lmhead_forward_noalloc: the fused LM-head forward for callers that
// cannot allocate device memory on demand.
//
// Those callers cannot hand slp_lmhead_forward the workspace it asks for.
// Their framework may own every byte of device memory through its own pool or
// budget, or the place they call from may not tolerate cudaMalloc, which
// synchronises the whole device.  This entry point takes its scratch from one
// fixed array in the library's device image instead.  The array is
// kStaticScratchBytes (16 MiB) on every GPU that loads the library and stays
// there until the process exits.
//
// Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library
// call.  The first call on a device looks the array up with
// cudaGetSymbolAddress while that device is current and caches the address;
// make that first call before any stream capture.  The cached address belongs
// to the device's current context: after a cudaDeviceReset it is stale, and
// the call must not be used on that device again.  Every call on a device
// uses the same array and leaves its contents behind.  No byte of it has to
// start at zero: every value the kernels read is written earlier in the same
// call.  Two calls whose work overlaps on the GPU (other streams, or a second
// call launched before the first finished) race on the array.

#include "slp.h"
#include "slp_internal.h"

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;

}  // namespace

static __device__ __align__(256) unsigned char slp_static_scratch[kStaticScratchBytes];

namespace {

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of slp_static_scratch on the current device (looked up once
// per device; the host-side symbol itself is not a device address).
cudaError_t static_scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, slp_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int slp_lmhead_forward_noalloc(const void* h, const void* W, int64_t N, int64_t V,
                                          int64_t d, const int32_t* t, const uint8_t* mask,
                                          float T, float* logprob, float* lse, int32_t* err,
                                          void* stream) {
  if (N < 0 || V <= 0 || d <= 0 || V > INT32_MAX || N > INT32_MAX || d > INT32_MAX)
    return SLP_ERR_INVALID_ARG;
  if (!(isfinite(T) && T > 0.f)) return SLP_ERR_INVALID_ARG;
  if (N == 0) return SLP_OK;
  if (h == nullptr || W == nullptr || t == nullptr || logprob == nullptr || lse == nullptr)
    return SLP_ERR_INVALID_ARG;
  if (d % 64 != 0) return SLP_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(h) & 15u) || (reinterpret_cast<uintptr_t>(W) & 15u))
    return SLP_ERR_MISALIGNED;
  if (slp::lmhead_forward_workspace_size(N, V, d) > kStaticScratchBytes) return SLP_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (static_scratch_for_current_device(&scratch) != cudaSuccess) return SLP_ERR_CUDA;
  const cudaError_t e = slp::launch_lmhead_forward(h, W, N, V, d, t, mask, T, logprob, lse,
                                                   scratch, err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SLP_OK : SLP_ERR_CUDA;
}
