// C-ABI entry points of libslp: argument validation (before any CUDA call, so
// argument errors are reported without touching the device), then the kernel
// launchers.  The library allocates nothing and never synchronises.

#include "slp.h"
#include "slp_bounds.cuh"
#include "slp_internal.h"

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

namespace slp {

int sm_count() {
  // per device, filled on first use; threads that race here store the same value
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace slp

namespace {

// One CTA whose bounds table holds buf[0..4) only: it loads and stores
// buf[4], which the bounds-checked build must refuse, and stores buf[0],
// which it must make.
__global__ void bounds_selftest_kernel(float* buf SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  if (threadIdx.x == 0) {
    const float v = slp::dbg::ld(buf + 4);
    slp::dbg::st(buf + 4, v + 1.0f);
    slp::dbg::st(buf, 1.0f);
  }
}

bool temperature_ok(float T) { return isfinite(T) && T > 0.f; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SLP_OK : SLP_ERR_CUDA; }

int check_logits_args(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                      const int32_t* t, float T) {
  if (dtype != SLP_BF16 && dtype != SLP_F32) return SLP_ERR_INVALID_ARG;
  if (N < 0 || V <= 0 || ld < V || V > INT32_MAX) return SLP_ERR_INVALID_ARG;
  if (!temperature_ok(T)) return SLP_ERR_INVALID_ARG;
  if (N > 0 && (x == nullptr || t == nullptr)) return SLP_ERR_INVALID_ARG;
  return SLP_OK;
}

int check_lmhead_args(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                      const int32_t* t, float T, void* ws, size_t ws_bytes, size_t ws_need) {
  if (N < 0 || V <= 0 || d <= 0 || V > INT32_MAX || N > INT32_MAX) return SLP_ERR_INVALID_ARG;
  if (!temperature_ok(T)) return SLP_ERR_INVALID_ARG;
  if (N == 0) return SLP_OK;
  if (h == nullptr || W == nullptr || t == nullptr) return SLP_ERR_INVALID_ARG;
  if (d % 64 != 0) return SLP_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(h) & 15u) || (reinterpret_cast<uintptr_t>(W) & 15u))
    return SLP_ERR_MISALIGNED;
  if (ws == nullptr || ws_bytes < ws_need) return SLP_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return SLP_ERR_MISALIGNED;
  return SLP_OK;
}

}  // namespace

extern "C" {

int slp_forward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld, const int32_t* t,
                const uint8_t* mask, float T, float* logprob, float* lse, int32_t* err,
                void* stream) {
  int st = check_logits_args(x, dtype, N, V, ld, t, T);
  if (st != SLP_OK) return st;
  if (N == 0) return SLP_OK;
  if (logprob == nullptr || lse == nullptr) return SLP_ERR_INVALID_ARG;
  return cuda_status(slp::launch_forward(x, dtype, N, V, ld, t, mask, T, logprob, lse, err,
                                         static_cast<cudaStream_t>(stream)));
}

int slp_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld, const int32_t* t,
                 const uint8_t* mask, float T, const float* lse, const float* grad_out,
                 void* grad_x, int64_t ld_grad, int32_t* err, void* stream) {
  int st = check_logits_args(x, dtype, N, V, ld, t, T);
  if (st != SLP_OK) return st;
  if (ld_grad < V) return SLP_ERR_INVALID_ARG;
  if (N == 0) return SLP_OK;
  if (lse == nullptr || grad_out == nullptr || grad_x == nullptr) return SLP_ERR_INVALID_ARG;
  return cuda_status(slp::launch_backward(x, dtype, N, V, ld, t, mask, T, lse, grad_out, grad_x,
                                          ld_grad, err, static_cast<cudaStream_t>(stream)));
}

int slp_forward_entropy(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                        const int32_t* t, const uint8_t* mask, float T, float* logprob,
                        float* lse, float* entropy, int32_t* err, void* stream) {
  int st = check_logits_args(x, dtype, N, V, ld, t, T);
  if (st != SLP_OK) return st;
  if (N == 0) return SLP_OK;
  if (logprob == nullptr || lse == nullptr || entropy == nullptr) return SLP_ERR_INVALID_ARG;
  return cuda_status(slp::launch_forward_entropy(x, dtype, N, V, ld, t, mask, T, logprob, lse,
                                                 entropy, err, static_cast<cudaStream_t>(stream)));
}

int slp_backward_entropy(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                         const int32_t* t, const uint8_t* mask, float T, const float* lse,
                         const float* entropy, const float* grad_out, const float* grad_entropy,
                         void* grad_x, int64_t ld_grad, int32_t* err, void* stream) {
  int st = check_logits_args(x, dtype, N, V, ld, t, T);
  if (st != SLP_OK) return st;
  if (ld_grad < V) return SLP_ERR_INVALID_ARG;
  if (N == 0) return SLP_OK;
  if (lse == nullptr || entropy == nullptr || grad_x == nullptr) return SLP_ERR_INVALID_ARG;
  return cuda_status(slp::launch_backward_entropy(x, dtype, N, V, ld, t, mask, T, lse, entropy,
                                                  grad_out, grad_entropy, grad_x, ld_grad, err,
                                                  static_cast<cudaStream_t>(stream)));
}

int slp_topk_kl_forward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                        const int32_t* ids, const float* teacher_logp, int64_t K,
                        const uint8_t* mask, float T, float clamp_min, float* kl,
                        float* student_mass, float* teacher_mass, float* lse, int32_t* err,
                        void* stream) {
  int st = check_logits_args(x, dtype, N, V, ld, ids, T);
  if (st != SLP_OK) return st;
  if (K < 1 || K > INT32_MAX / 2 || isnan(clamp_min)) return SLP_ERR_INVALID_ARG;
  if (N == 0) return SLP_OK;
  if (teacher_logp == nullptr || kl == nullptr || student_mass == nullptr ||
      teacher_mass == nullptr || lse == nullptr)
    return SLP_ERR_INVALID_ARG;
  return cuda_status(slp::launch_topk_kl_forward(x, dtype, N, V, ld, ids, teacher_logp, K, mask,
                                                 T, clamp_min, kl, student_mass, teacher_mass,
                                                 lse, err, static_cast<cudaStream_t>(stream)));
}

int slp_topk_kl_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                         const int32_t* ids, const float* teacher_logp, int64_t K,
                         const uint8_t* mask, float T, float clamp_min, const float* lse,
                         const float* grad_kl, void* grad_x, int64_t ld_grad, int32_t* err,
                         void* stream) {
  int st = check_logits_args(x, dtype, N, V, ld, ids, T);
  if (st != SLP_OK) return st;
  if (K < 1 || K > INT32_MAX / 2 || isnan(clamp_min) || ld_grad < V) return SLP_ERR_INVALID_ARG;
  if (K > slp::topk_kl_max_k()) return SLP_ERR_UNSUPPORTED;
  if (N == 0) return SLP_OK;
  if (teacher_logp == nullptr || lse == nullptr || grad_kl == nullptr || grad_x == nullptr)
    return SLP_ERR_INVALID_ARG;
  return cuda_status(slp::launch_topk_kl_backward(x, dtype, N, V, ld, ids, teacher_logp, K, mask,
                                                  T, clamp_min, lse, grad_kl, grad_x, ld_grad,
                                                  err, static_cast<cudaStream_t>(stream)));
}

int slp_forward_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                         const int32_t* t, const uint8_t* mask, float T, const float* grad_out,
                         float* logprob, float* lse, void* grad_x, int64_t ld_grad, int32_t* err,
                         void* stream) {
  int st = check_logits_args(x, dtype, N, V, ld, t, T);
  if (st != SLP_OK) return st;
  if (ld_grad < V) return SLP_ERR_INVALID_ARG;
  if (N == 0) return SLP_OK;
  if (grad_out == nullptr || logprob == nullptr || lse == nullptr || grad_x == nullptr)
    return SLP_ERR_INVALID_ARG;
  return cuda_status(slp::launch_forward_backward(x, dtype, N, V, ld, t, mask, T, grad_out,
                                                  logprob, lse, grad_x, ld_grad, err,
                                                  static_cast<cudaStream_t>(stream)));
}

int slp_forward_backward_entropy(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                 const int32_t* t, const uint8_t* mask, float T,
                                 const float* grad_out, const float* grad_entropy, float* logprob,
                                 float* lse, float* entropy, void* grad_x, int64_t ld_grad,
                                 int32_t* err, void* stream) {
  int st = check_logits_args(x, dtype, N, V, ld, t, T);
  if (st != SLP_OK) return st;
  if (ld_grad < V) return SLP_ERR_INVALID_ARG;
  if (N == 0) return SLP_OK;
  if (logprob == nullptr || lse == nullptr || entropy == nullptr || grad_x == nullptr)
    return SLP_ERR_INVALID_ARG;
  return cuda_status(slp::launch_forward_backward_entropy(
      x, dtype, N, V, ld, t, mask, T, grad_out, grad_entropy, logprob, lse, entropy, grad_x,
      ld_grad, err, static_cast<cudaStream_t>(stream)));
}

size_t slp_forward_backward_host_workspace_size(int64_t N, int64_t V, int dtype,
                                                int64_t rows_per_chunk) {
  if (N < 0 || V <= 0 || V > INT32_MAX || (dtype != SLP_BF16 && dtype != SLP_F32)) return 0;
  return slp::forward_backward_host_workspace_size(N, V, dtype == SLP_BF16 ? 2 : 4,
                                                   rows_per_chunk);
}

int slp_forward_backward_host(const void* x_host, int dtype, int64_t N, int64_t V, int64_t ld,
                              const int32_t* t_host, const uint8_t* mask_host, float T,
                              const float* g_host, float* logprob_host, float* lse_host,
                              void* grad_x_host, int64_t ld_grad, int64_t rows_per_chunk,
                              void* ws, size_t ws_bytes, int32_t* err, void* stream) {
  int st = check_logits_args(x_host, dtype, N, V, ld, t_host, T);
  if (st != SLP_OK) return st;
  if (ld_grad < V) return SLP_ERR_INVALID_ARG;
  if (N == 0) return SLP_OK;
  if (g_host == nullptr || logprob_host == nullptr || lse_host == nullptr || grad_x_host == nullptr)
    return SLP_ERR_INVALID_ARG;
  // every host buffer must be page-locked (asynchronous copies)
  const void* host_ptrs[7] = {x_host, t_host, mask_host, g_host, logprob_host, lse_host,
                              grad_x_host};
  for (const void* hp : host_ptrs) {
    if (hp == nullptr) continue;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, hp) != cudaSuccess) {
      cudaGetLastError();
      return SLP_ERR_INVALID_ARG;
    }
    if (a.type != cudaMemoryTypeHost) return SLP_ERR_INVALID_ARG;
  }
  const size_t need = slp::forward_backward_host_workspace_size(
      N, V, dtype == SLP_BF16 ? 2 : 4, rows_per_chunk);
  if (ws == nullptr || ws_bytes < need) return SLP_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return SLP_ERR_MISALIGNED;
  return cuda_status(slp::launch_forward_backward_host(
      x_host, dtype, N, V, ld, t_host, mask_host, T, g_host, logprob_host, lse_host, grad_x_host,
      ld_grad, rows_per_chunk, ws, err, static_cast<cudaStream_t>(stream)));
}

size_t slp_lmhead_workspace_size(int64_t N, int64_t V, int64_t d) {
  if (N < 0 || V <= 0 || d <= 0 || V > INT32_MAX || N > INT32_MAX || d > INT32_MAX) return 0;
  return slp::lmhead_workspace_size(N, V, d);
}

size_t slp_lmhead_workspace_size_max(int64_t N, int64_t V, int64_t d) {
  if (N < 0 || V <= 0 || d <= 0 || V > INT32_MAX || N > INT32_MAX || d > INT32_MAX) return 0;
  return slp::lmhead_workspace_size_max(N, V, d);
}

size_t slp_lmhead_workspace_size_min(int64_t N, int64_t V, int64_t d) {
  if (N < 0 || V <= 0 || d <= 0 || V > INT32_MAX || N > INT32_MAX || d > INT32_MAX) return 0;
  return slp::lmhead_workspace_size_min(N, V, d);
}

size_t slp_lmhead_forward_workspace_size(int64_t N, int64_t V, int64_t d) {
  if (N < 0 || V <= 0 || d <= 0 || V > INT32_MAX || N > INT32_MAX || d > INT32_MAX) return 0;
  return slp::lmhead_forward_workspace_size(N, V, d);
}

int slp_lmhead_forward(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                       const int32_t* t, const uint8_t* mask, float T, float* logprob,
                       float* lse, void* ws, size_t ws_bytes, int32_t* err, void* stream) {
  int st = check_lmhead_args(h, W, N, V, d, t, T, ws, ws_bytes,
                             slp::lmhead_forward_workspace_size(N, V, d));
  if (st != SLP_OK) return st;
  if (N == 0) return SLP_OK;
  if (logprob == nullptr || lse == nullptr) return SLP_ERR_INVALID_ARG;
  return cuda_status(slp::launch_lmhead_forward(h, W, N, V, d, t, mask, T, logprob, lse, ws, err,
                                                static_cast<cudaStream_t>(stream)));
}

int slp_lmhead_backward(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                        const int32_t* t, const uint8_t* mask, float T, const float* lse,
                        const float* grad_out, void* dh, void* dW, void* ws, size_t ws_bytes,
                        int32_t* err, void* stream) {
  int st = check_lmhead_args(h, W, N, V, d, t, T, ws, ws_bytes,
                             slp::lmhead_workspace_size_min(N, V, d));
  if (st != SLP_OK) return st;
  if (N == 0) return SLP_OK;
  if (lse == nullptr || grad_out == nullptr || dh == nullptr || dW == nullptr)
    return SLP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dh) & 15u) || (reinterpret_cast<uintptr_t>(dW) & 15u))
    return SLP_ERR_MISALIGNED;
  return cuda_status(slp::launch_lmhead_backward(h, W, N, V, d, t, mask, T, lse, grad_out, dh,
                                                 dW, ws, ws_bytes, err,
                                                 static_cast<cudaStream_t>(stream)));
}

int slp_lmhead_backward_accumulate(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                                   const int32_t* t, const uint8_t* mask, float T,
                                   const float* lse, const float* grad_out, void* dh,
                                   float* dW_accum, void* ws, size_t ws_bytes, int32_t* err,
                                   void* stream) {
  int st = check_lmhead_args(h, W, N, V, d, t, T, ws, ws_bytes,
                             slp::lmhead_workspace_size_min(N, V, d));
  if (st != SLP_OK) return st;
  if (N == 0) return SLP_OK;
  if (lse == nullptr || grad_out == nullptr || dh == nullptr || dW_accum == nullptr)
    return SLP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dh) & 15u) || (reinterpret_cast<uintptr_t>(dW_accum) & 15u))
    return SLP_ERR_MISALIGNED;
  return cuda_status(slp::launch_lmhead_backward(h, W, N, V, d, t, mask, T, lse, grad_out, dh,
                                                 dW_accum, ws, ws_bytes, err,
                                                 static_cast<cudaStream_t>(stream), true));
}

uint64_t slp_lmhead_set_wait_limit_ns(uint64_t ns) { return slp::lmhead_set_wait_limit(ns); }

int slp_bounds_check_selftest(float* buf, int32_t* err, void* stream) {
#ifdef SLP_DEBUG_BOUNDS
  if (buf == nullptr || err == nullptr) return SLP_ERR_INVALID_ARG;
  bounds_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      buf SLP_DBG_ARG(err, {{buf, 16ull}}));
  return cuda_status(cudaGetLastError());
#else
  (void)buf;
  (void)err;
  (void)stream;
  return SLP_ERR_UNSUPPORTED;
#endif
}

const char* slp_status_string(int status) {
  switch (status) {
    case SLP_OK: return "ok";
    case SLP_ERR_INVALID_ARG: return "invalid argument";
    case SLP_ERR_UNSUPPORTED: return "unsupported shape";
    case SLP_ERR_MISALIGNED: return "misaligned pointer or stride";
    case SLP_ERR_WORKSPACE: return "workspace missing or too small";
    case SLP_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

}  // extern "C"
