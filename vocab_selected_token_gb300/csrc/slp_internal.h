// Internal interface between the C-ABI layer (slp_api.cu) and the kernel
// launchers.  Arguments have been validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace slp {

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Logits-input path (slp_logits.cu).
cudaError_t launch_forward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                           const int32_t* t, const uint8_t* mask, float T, float* logprob,
                           float* lse, int32_t* err, cudaStream_t stream);

cudaError_t launch_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                            const int32_t* t, const uint8_t* mask, float T, const float* lse,
                            const float* grad_out, void* grad_x, int64_t ld_grad,
                            int32_t* err, cudaStream_t stream);

cudaError_t launch_forward_entropy(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                   const int32_t* t, const uint8_t* mask, float T,
                                   float* logprob, float* lse, float* entropy, int32_t* err,
                                   cudaStream_t stream);

cudaError_t launch_backward_entropy(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                    const int32_t* t, const uint8_t* mask, float T,
                                    const float* lse, const float* entropy,
                                    const float* grad_out, const float* grad_entropy,
                                    void* grad_x, int64_t ld_grad, int32_t* err,
                                    cudaStream_t stream);

cudaError_t launch_forward_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                    const int32_t* t, const uint8_t* mask, float T,
                                    const float* grad_out, float* logprob, float* lse,
                                    void* grad_x, int64_t ld_grad, int32_t* err,
                                    cudaStream_t stream);

cudaError_t launch_forward_backward_entropy(const void* x, int dtype, int64_t N, int64_t V,
                                            int64_t ld, const int32_t* t, const uint8_t* mask,
                                            float T, const float* grad_out,
                                            const float* grad_entropy, float* logprob, float* lse,
                                            float* entropy, void* grad_x, int64_t ld_grad,
                                            int32_t* err, cudaStream_t stream);

// Host-resident logits streamed through slp_forward_backward (slp_host.cu).
size_t forward_backward_host_workspace_size(int64_t N, int64_t V, int esize,
                                            int64_t rows_per_chunk);
cudaError_t launch_forward_backward_host(const void* x_host, int dtype, int64_t N, int64_t V,
                                         int64_t ld, const int32_t* t_host,
                                         const uint8_t* mask_host, float T, const float* g_host,
                                         float* lp_host, float* lse_host, void* gx_host,
                                         int64_t ld_grad, int64_t rows_per_chunk, void* ws,
                                         int32_t* err, cudaStream_t stream);

// Top-k forward KL (slp_topk.cu).
int64_t topk_kl_max_k();
cudaError_t launch_topk_kl_forward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                   const int32_t* ids, const float* teacher_logp, int64_t K,
                                   const uint8_t* mask, float T, float clamp_min, float* kl,
                                   float* student_mass, float* teacher_mass, float* lse,
                                   int32_t* err, cudaStream_t stream);
cudaError_t launch_topk_kl_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                    const int32_t* ids, const float* teacher_logp, int64_t K,
                                    const uint8_t* mask, float T, float clamp_min,
                                    const float* lse, const float* grad_kl, void* grad_x,
                                    int64_t ld_grad, int32_t* err, cudaStream_t stream);

// Fused LM-head path (slp_lmhead.cu).
size_t lmhead_workspace_size(int64_t N, int64_t V, int64_t d);
size_t lmhead_workspace_size_max(int64_t N, int64_t V, int64_t d);
size_t lmhead_workspace_size_min(int64_t N, int64_t V, int64_t d);
size_t lmhead_forward_workspace_size(int64_t N, int64_t V, int64_t d);
// Sets the bound of every pipeline wait in later LM-head launches (0: the
// default of two seconds); returns the previous bound.
uint64_t lmhead_set_wait_limit(uint64_t ns);

cudaError_t launch_lmhead_forward(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                                  const int32_t* t, const uint8_t* mask, float T,
                                  float* logprob, float* lse, void* ws, int32_t* err,
                                  cudaStream_t stream);

cudaError_t launch_lmhead_backward(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                                   const int32_t* t, const uint8_t* mask, float T,
                                   const float* lse, const float* grad_out, void* dh, void* dW,
                                   void* ws, size_t ws_bytes, int32_t* err, cudaStream_t stream,
                                   bool accumulate_f32 = false);

}  // namespace slp
