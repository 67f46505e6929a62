// Chunked top-k forward KL on the same log-sum-exp engine (verl PR #7733
// "memory-efficient chunked top-k KL", "Design & Code Changes": the teacher
// is given by its top-k ids and log-probabilities; the student's global logZ
// comes from a max/sum pass over its logits; backward recomputes the student
// probabilities from the saved logZ instead of storing them).
//
//   ls[k] = x[ids[k]] / T - lse,  lc[k] = max(ls[k], clamp_min),  p[k] = exp(lt[k])
//   kl = sum_k p[k] (lt[k] - lc[k]);  student_mass = sum_k exp(ls[k]);
//   teacher_mass = sum_k p[k]
//   grad_x[v] = g / T * ( P q[v] - sum_{k: ids[k] = v, ls[k] >= clamp} p[k] ),
//   P = sum of the kept p[k],  q = softmax(x / T).
//
// Forward: the streaming log-sum-exp kernel of the logits path (no target),
// then one warp per row over the K teacher entries.  Backward: one CTA per
// row streams the row once, writing the dense part g/T P q[v]; a bitmap of the
// row's teacher ids in shared memory flags the few elements that also take a
// -g/T p[k] term, so the sparse part costs one shared-memory word test per
// eight elements.

#include "slp.h"
#include "slp_device.cuh"
#include "slp_internal.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace slp {
namespace {

constexpr int kTkThreads = 256;
constexpr int kTkUnroll = 4;
constexpr int kTkMaxSmem = 160 * 1024;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

template <typename Elt>
__global__ void __launch_bounds__(256)
    slp_topk_kl_rows_kernel(const Elt* __restrict__ x, int64_t N, int64_t V, int64_t ld,
                            const int32_t* __restrict__ ids, const float* __restrict__ lt, int K,
                            const uint8_t* __restrict__ mask, float invT, float clamp_min,
                            const float* __restrict__ lse, float* __restrict__ kl,
                            float* __restrict__ smass, float* __restrict__ tmass,
                            int32_t* __restrict__ err) {
  using E = Elem<Elt>;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= N) return;
  if (mask != nullptr && mask[row] == 0) {
    if (lane == 0) kl[row] = smass[row] = tmass[row] = 0.f;
    return;
  }
  const float L = lse[row];
  const Elt* xr = x + row * ld;
  float a_kl = 0.f, a_sm = 0.f, a_tm = 0.f;
  bool bad = false;
  for (int k = lane; k < K; k += 32) {
    const int id = ids[row * K + k];
    if (id < 0 || static_cast<int64_t>(id) >= V) {
      bad = true;
      continue;
    }
    const float ls = fmaf(E::load1(xr + id), invT, -L);
    const float tk = lt[row * K + k];
    const float p = expf(tk);
    a_kl = fmaf(p, tk - fmaxf(ls, clamp_min), a_kl);
    a_sm += expf(ls);
    a_tm += p;
  }
  a_kl = warp_sum(a_kl);
  a_sm = warp_sum(a_sm);
  a_tm = warp_sum(a_tm);
  bad = __any_sync(0xFFFFFFFFu, bad);
  if (lane == 0) {
    if (bad) {
      if (err != nullptr) atomicOr(err, SLP_DATA_ERR_TARGET);
      a_kl = a_sm = a_tm = __int_as_float(0x7FC00000);
    }
    kl[row] = a_kl;
    smass[row] = a_sm;
    tmass[row] = a_tm;
  }
}

template <typename Elt, bool kVecPath>
__global__ void __launch_bounds__(kTkThreads)
    slp_topk_kl_bwd_kernel(const Elt* __restrict__ x, int64_t V, int64_t ld,
                           const int32_t* __restrict__ ids, const float* __restrict__ lt, int K,
                           const uint8_t* __restrict__ mask, float invT, float c,
                           float clamp_min, const float* __restrict__ lse,
                           const float* __restrict__ g, Elt* __restrict__ gx, int64_t ldg,
                           int32_t* __restrict__ err) {
  using E = Elem<Elt>;
  constexpr int kVec = E::kVec;
  extern __shared__ uint32_t tk_smem[];
  __shared__ float warp_p[kTkThreads / 32];
  const int64_t row = blockIdx.x;
  const Elt* xr = x + row * ld;
  Elt* gr = gx + row * ldg;
  const int64_t nvec = kVecPath ? V / kVec : 0;

  if (mask != nullptr && mask[row] == 0) {
    if (kVecPath) {
      uint4* gv = reinterpret_cast<uint4*>(gr);
      for (int64_t i = threadIdx.x; i < nvec; i += kTkThreads) st_stream(gv + i, make_uint4(0, 0, 0, 0));
    }
    for (int64_t e = nvec * kVec + threadIdx.x; e < V; e += kTkThreads) E::store1(gr + e, 0.f);
    return;
  }

  const int nwords = static_cast<int>((V + 31) / 32);
  uint32_t* bitmap = tk_smem;
  int* sid = reinterpret_cast<int*>(bitmap + nwords);
  float* sp = reinterpret_cast<float*>(sid + K);
  for (int w = threadIdx.x; w < nwords; w += kTkThreads) bitmap[w] = 0u;
  __syncthreads();

  const float L = lse[row];
  float gT = g[row] * invT;
  float pl = 0.f;
  bool bad = false;
  for (int k = threadIdx.x; k < K; k += kTkThreads) {
    const int id = ids[row * K + k];
    float p = 0.f;
    if (id < 0 || static_cast<int64_t>(id) >= V) {
      bad = true;
      sid[k] = -1;
    } else {
      const float ls = fmaf(E::load1(xr + id), invT, -L);
      p = ls >= clamp_min ? expf(lt[row * K + k]) : 0.f;
      sid[k] = id;
      atomicOr(&bitmap[id >> 5], 1u << (id & 31));
    }
    sp[k] = p;
    pl += p;
  }
  // P in a fixed order: lane sums, then warps in order
  pl = warp_sum(pl);
  if ((threadIdx.x & 31) == 0) warp_p[threadIdx.x >> 5] = pl;
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0 && err != nullptr) atomicOr(err, SLP_DATA_ERR_TARGET);
    gT = __int_as_float(0x7FC00000);
  }
  float P = 0.f;
#pragma unroll
  for (int w = 0; w < kTkThreads / 32; ++w) P += warp_p[w];
  const float dense = gT * P;
  const float L2 = L * kLog2e;

  // teacher mass sitting on element v (kept entries; ids may repeat)
  auto sparse = [&](int64_t v) {
    float s = 0.f;
    for (int k = 0; k < K; ++k)
      if (sid[k] == v) s += sp[k];
    return s;
  };
  auto marked = [&](int64_t v) { return (bitmap[v >> 5] >> (v & 31)) & 1u; };

  if constexpr (kVecPath) {
    const uint4* xv = reinterpret_cast<const uint4*>(xr);
    uint4* gv = reinterpret_cast<uint4*>(gr);
    for (int64_t i0 = threadIdx.x; i0 < nvec; i0 += kTkThreads * kTkUnroll) {
      uint4 buf[kTkUnroll];
#pragma unroll
      for (int u = 0; u < kTkUnroll; ++u) {
        const int64_t i = i0 + static_cast<int64_t>(u) * kTkThreads;
        if (i < nvec) buf[u] = ld_stream(xv + i);
      }
#pragma unroll
      for (int u = 0; u < kTkUnroll; ++u) {
        const int64_t i = i0 + static_cast<int64_t>(u) * kTkThreads;
        if (i < nvec) {
          float f[kVec];
          E::unpack(buf[u], f);
#pragma unroll
          for (int j = 0; j < kVec; ++j) f[j] = dense * ex2(fmaf(f[j], c, -L2));
          // the kVec elements of vector i share one bitmap word
          const int64_t e0 = i * kVec;
          const uint32_t bits = (bitmap[e0 >> 5] >> (e0 & 31)) & ((1u << kVec) - 1u);
          if (bits != 0u) {
#pragma unroll
            for (int j = 0; j < kVec; ++j)
              if ((bits >> j) & 1u) f[j] = fmaf(-gT, sparse(e0 + j), f[j]);
          }
          st_stream(gv + i, E::pack(f));
        }
      }
    }
  }
  for (int64_t e = nvec * kVec + threadIdx.x; e < V; e += kTkThreads) {
    float o = dense * ex2(fmaf(E::load1(xr + e), c, -L2));
    if (marked(e)) o = fmaf(-gT, sparse(e), o);
    E::store1(gr + e, o);
  }
}

bool aligned16(const void* p, int64_t ld, int esize) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ((ld * esize) & 15) == 0;
}

template <typename Elt>
cudaError_t topk_bwd_typed(const Elt* x, int64_t N, int64_t V, int64_t ld, const int32_t* ids,
                           const float* lt, int K, const uint8_t* mask, float T, float clamp_min,
                           const float* lse, const float* g, Elt* gx, int64_t ldg, int32_t* err,
                           cudaStream_t stream) {
  const int64_t smem = (V + 31) / 32 * 4 + static_cast<int64_t>(K) * 8;
  if (smem > kTkMaxSmem || N > 0x7FFFFFFFLL) return cudaErrorNotSupported;
  const float invT = 1.0f / T;
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  const bool vec = aligned16(x, ld, sizeof(Elt)) && aligned16(gx, ldg, sizeof(Elt));
  auto k = vec ? slp_topk_kl_bwd_kernel<Elt, true> : slp_topk_kl_bwd_kernel<Elt, false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kTkMaxSmem);
  if (e != cudaSuccess) return e;
  k<<<static_cast<unsigned>(N), kTkThreads, static_cast<size_t>(smem), stream>>>(
      x, V, ld, ids, lt, K, mask, invT, c, clamp_min, lse, g, gx, ldg, err);
  return cudaGetLastError();
}

}  // namespace

size_t topk_kl_max_vocab(int64_t K) {
  const int64_t words = (kTkMaxSmem - K * 8) / 4;
  return words > 0 ? static_cast<size_t>(words * 32) : 0;
}

cudaError_t launch_topk_kl_forward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                   const int32_t* ids, const float* teacher_logp, int64_t K,
                                   const uint8_t* mask, float T, float clamp_min, float* kl,
                                   float* student_mass, float* teacher_mass, float* lse,
                                   int32_t* err, cudaStream_t stream) {
  cudaError_t e = launch_forward(x, dtype, N, V, ld, nullptr, mask, T, nullptr, lse, err, stream);
  if (e != cudaSuccess) return e;
  const unsigned blocks = static_cast<unsigned>((N + 7) / 8);
  const float invT = 1.0f / T;
  if (dtype == SLP_BF16)
    slp_topk_kl_rows_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(x), N, V, ld, ids, teacher_logp, static_cast<int>(K),
        mask, invT, clamp_min, lse, kl, student_mass, teacher_mass, err);
  else
    slp_topk_kl_rows_kernel<float><<<blocks, 256, 0, stream>>>(
        static_cast<const float*>(x), N, V, ld, ids, teacher_logp, static_cast<int>(K), mask,
        invT, clamp_min, lse, kl, student_mass, teacher_mass, err);
  return cudaGetLastError();
}

cudaError_t launch_topk_kl_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                    const int32_t* ids, const float* teacher_logp, int64_t K,
                                    const uint8_t* mask, float T, float clamp_min,
                                    const float* lse, const float* grad_kl, void* grad_x,
                                    int64_t ld_grad, int32_t* err, cudaStream_t stream) {
  if (dtype == SLP_BF16)
    return topk_bwd_typed(static_cast<const __nv_bfloat16*>(x), N, V, ld, ids, teacher_logp,
                          static_cast<int>(K), mask, T, clamp_min, lse, grad_kl,
                          static_cast<__nv_bfloat16*>(grad_x), ld_grad, err, stream);
  return topk_bwd_typed(static_cast<const float*>(x), N, V, ld, ids, teacher_logp,
                        static_cast<int>(K), mask, T, clamp_min, lse, grad_kl,
                        static_cast<float*>(grad_x), ld_grad, err, stream);
}

}  // namespace slp
