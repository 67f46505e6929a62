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
// row streams the row once through a bulk-copy ring, writing the dense part
// g/T P q[v] everywhere; then the K elements that carry teacher entries are
// rewritten in full (recomputed in fp32 and rounded once), so the streaming
// pass stays a plain elementwise pass.  Rows of at most 32 KB (with K <= 256)
// take the same backward with one warp per row.

#include "slp.h"
#include "slp_device.cuh"
#include "slp_internal.h"
#include "slp_sm100.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace slp {
namespace {

constexpr int kTkThreads = 256;
constexpr int kTkStages = 4;     // bulk-copy ring of the vector path
constexpr int kTkChunk = 16384;  // bytes per copy: 4 vectors per thread
constexpr int kTkRing = kTkStages * kTkChunk;
constexpr int kTkMaxSmem = 128 * 1024;  // teacher entries (8 bytes each)
constexpr uint64_t kTkWaitNs = 2000000000ull;

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
                            int32_t* __restrict__ err SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  using E = Elem<Elt>;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= N) return;
  if (mask != nullptr && dbg::ld(mask + row) == 0) {
    if (lane == 0) {
      dbg::st(kl + row, 0.f);
      dbg::st(smass + row, 0.f);
      dbg::st(tmass + row, 0.f);
    }
    return;
  }
  const float L = dbg::ld(lse + row);
  const Elt* xr = x + row * ld;
  float a_kl = 0.f, a_sm = 0.f, a_tm = 0.f;
  bool bad = false;
  for (int k = lane; k < K; k += 32) {
    const int id = dbg::ld(ids + row * K + k);
    if (id < 0 || static_cast<int64_t>(id) >= V) {
      bad = true;
      continue;
    }
    const float ls = fmaf(E::load1(xr + id), invT, -L);
    const float tk = dbg::ld(lt + row * K + k);
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
    dbg::st(kl + row, a_kl);
    dbg::st(smass + row, a_sm);
    dbg::st(tmass + row, a_tm);
  }
}

template <typename Elt, bool kVecPath>
__global__ void __launch_bounds__(kTkThreads)
    slp_topk_kl_bwd_kernel(const Elt* __restrict__ x, int64_t V, int64_t ld,
                           const int32_t* __restrict__ ids, const float* __restrict__ lt, int K,
                           const uint8_t* __restrict__ mask, float invT, float c,
                           float clamp_min, const float* __restrict__ lse,
                           const float* __restrict__ g, Elt* __restrict__ gx, int64_t ldg,
                           int32_t* __restrict__ err SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  using E = Elem<Elt>;
  constexpr int kVec = E::kVec;
  extern __shared__ __align__(128) uint8_t tk_smem[];
  __shared__ float warp_p[kTkThreads / 32];
  const int64_t row = blockIdx.x;
  const Elt* xr = x + row * ld;
  Elt* gr = gx + row * ldg;
  const int64_t nvec = kVecPath ? V / kVec : 0;

  if (mask != nullptr && dbg::ld(mask + row) == 0) {
    if (kVecPath) {
      uint4* gv = reinterpret_cast<uint4*>(gr);
      for (int64_t i = threadIdx.x; i < nvec; i += kTkThreads) st_stream(gv + i, make_uint4(0, 0, 0, 0));
    }
    for (int64_t e = nvec * kVec + threadIdx.x; e < V; e += kTkThreads) E::store1(gr + e, 0.f);
    return;
  }

  // teacher entries: id, kept probability p (0 where the clamp is active)
  uint8_t* ring = tk_smem;                                        // kTkRing bytes (vector path)
  int* sid = reinterpret_cast<int*>(tk_smem + (kVecPath ? kTkRing : 0));
  float* sp = reinterpret_cast<float*>(sid + K);
  const float L = dbg::ld(lse + row);
  const float L2 = L * kLog2e;
  float gT = dbg::ld(g + row) * invT;
  float pl = 0.f;
  bool bad = false;
  for (int k = threadIdx.x; k < K; k += kTkThreads) {
    const int id = dbg::ld(ids + row * K + k);
    float p = 0.f;
    if (id < 0 || static_cast<int64_t>(id) >= V) {
      bad = true;
      sid[k] = -1;
    } else {
      const float ls = fmaf(E::load1(xr + id), invT, -L);
      p = ls >= clamp_min ? expf(dbg::ld(lt + row * K + k)) : 0.f;
      sid[k] = id;
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

  // pass 1: the dense part g/T P q[v] for every element
  if constexpr (kVecPath) {
    __shared__ __align__(8) uint64_t full[kTkStages];
    __shared__ int abort_flag;
    const char* src = reinterpret_cast<const char*>(xr);
    const int64_t nbytes = nvec * 16;
    const int64_t nch = (nbytes + kTkChunk - 1) / kTkChunk;
    const uint32_t sbase = sm100::smem_u32(ring);
    const uint32_t bbase = sm100::smem_u32(full);
    if (threadIdx.x == 0) {
      for (int st = 0; st < kTkStages; ++st) sm100::mbar_init(bbase + 8 * st, 1);
      abort_flag = 0;
      sm100::fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int64_t ch) {
      const int st = static_cast<int>(ch % kTkStages);
      const int64_t off = ch * kTkChunk;
      const uint32_t bytes = static_cast<uint32_t>(
          nbytes - off < kTkChunk ? nbytes - off : static_cast<int64_t>(kTkChunk));
      sm100::mbar_arrive_expect_tx(bbase + 8 * st, bytes);
      sm100::bulk_load(sbase + st * kTkChunk, src + off, bytes, bbase + 8 * st);
    };
    if (threadIdx.x == 0)
      for (int64_t ch = 0; ch < kTkStages && ch < nch; ++ch) issue(ch);
    uint4* gv = reinterpret_cast<uint4*>(gr);
    constexpr int kPer = kTkChunk / 16 / kTkThreads;
    const Elt* tag = nullptr;
    const float2 cc = make_float2(c, c);
    const float no1 = log2f(fabsf(dense)) - L2;
    const float2 no = make_float2(no1, no1);
    const uint32_t sgn = sign_mask(dense, tag);
    int64_t ch = 0;
    for (; ch < nch; ++ch) {
      const int st = static_cast<int>(ch % kTkStages);
      const bool got = sm100::mbar_wait_bounded(bbase + 8 * st, (ch / kTkStages) & 1,
                                                &abort_flag, kTkWaitNs);
      if (__syncthreads_or(!got)) break;
      const int64_t off = ch * kTkChunk;
      const int nv = static_cast<int>(
          (nbytes - off < kTkChunk ? nbytes - off : static_cast<int64_t>(kTkChunk)) / 16);
      const uint4* q = reinterpret_cast<const uint4*>(ring + st * kTkChunk);
      uint4 vv[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = u * kTkThreads + threadIdx.x;
        if (i < nv) vv[u] = q[i];
      }
      sm100::fence_proxy_async_smem();  // these reads precede the refill below
      __syncthreads();  // stage read: refill it while this chunk is written
      if (threadIdx.x == 0 && ch + kTkStages < nch) issue(ch + kTkStages);
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = u * kTkThreads + threadIdx.x;
        if (i < nv)  // dense * 2^(x c - L2) = sign(dense) 2^(x c - L2 + log2 |dense|)
          st_stream(gv + off / 16 + i, scaled_exp2_vec(vv[u], cc, no, sgn, tag));
      }
    }
    if (ch < nch) {
      if (threadIdx.x == 0) {
        if (err != nullptr) atomicOr(err, SLP_DEVICE_ERR_TIMEOUT);
        const int64_t last = ch + kTkStages < nch ? ch + kTkStages : nch;
        for (int64_t j = ch; j < last; ++j)
          sm100::mbar_wait_bounded(bbase + 8 * (j % kTkStages), (j / kTkStages) & 1, nullptr,
                                   kTkWaitNs);
      }
      __syncthreads();
    }
  }
  for (int64_t e = nvec * kVec + threadIdx.x; e < V; e += kTkThreads)
    E::store1(gr + e, dense * ex2(fmaf(E::load1(xr + e), c, -L2)));

  // pass 2: the elements carrying teacher entries, rewritten in full:
  // g/T (P q[v] - sum of the kept p over every entry with that id).  The first
  // entry of each id writes; the barrier orders it after pass 1's store.
  __syncthreads();
  for (int k = threadIdx.x; k < K; k += kTkThreads) {
    const int id = sid[k];
    if (id < 0) continue;
    bool first = true;
    float tot = 0.f;
    for (int j = 0; j < K; ++j) {
      if (sid[j] == id) {
        if (j < k) first = false;
        tot += sp[j];
      }
    }
    if (first) {
      const float q = ex2(fmaf(E::load1(xr + id), c, -L2));
      E::store1(gr + id, gT * fmaf(P, q, -tot));
    }
  }
}

// Short rows: the backward with one warp per row.  A CTA per row spends
// longer on its set-up (ring barriers, the K-entry table, CTA barriers) than
// on a row of a few KB.  Each warp keeps its row's K teacher entries (id,
// kept p) in its own slot of shared memory, padded to K4 = K rounded up to 4
// with id -2, streams the dense part with 16-byte loads (kTkRowsUnroll per
// lane in flight), then rewrites the elements that carry teacher entries as
// the CTA kernel does (same sums in the same order).  The search for other
// entries with the same id, K^2 / 32 steps per lane, reads the table four
// ids at a time.
constexpr int kTkRowsWarps = 8;
constexpr int kTkRowsUnroll = 8;
constexpr int kTkRowsMaxK = 256;  // 2 KB of entries per warp

template <typename Elt>
__global__ void __launch_bounds__(32 * kTkRowsWarps)
    slp_topk_kl_bwd_rows_kernel(const Elt* __restrict__ x, int64_t N, int64_t V, int64_t ld,
                                const int32_t* __restrict__ ids, const float* __restrict__ lt,
                                int K, const uint8_t* __restrict__ mask, float invT, float c,
                                float clamp_min, const float* __restrict__ lse,
                                const float* __restrict__ g, Elt* __restrict__ gx, int64_t ldg,
                                int32_t* __restrict__ err SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  using E = Elem<Elt>;
  constexpr int kVec = E::kVec;
  extern __shared__ __align__(16) int tk_rows_smem[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kTkRowsWarps + w;
  if (row >= N) return;
  const Elt* xr = x + row * ld;
  Elt* gr = gx + row * ldg;
  uint4* gv = reinterpret_cast<uint4*>(gr);
  const int64_t nvec = V / kVec;
  if (mask != nullptr && dbg::ld(mask + row) == 0) {
    for (int64_t i = lane; i < nvec; i += 32) st_stream(gv + i, make_uint4(0, 0, 0, 0));
    for (int64_t e = nvec * kVec + lane; e < V; e += 32) E::store1(gr + e, 0.f);
    return;
  }
  const int K4 = (K + 3) & ~3;
  int* sid = tk_rows_smem + static_cast<int64_t>(w) * 2 * K4;
  float* sp = reinterpret_cast<float*>(sid + K4);
  for (int k = K + lane; k < K4; k += 32) {
    sid[k] = -2;
    sp[k] = 0.f;
  }
  // the first batch of the dense pass is loaded before the entries are
  // gathered, so its latency overlaps the gather's dependent loads
  const uint4* xv = reinterpret_cast<const uint4*>(xr);
  uint4 v[kTkRowsUnroll];
#pragma unroll
  for (int u = 0; u < kTkRowsUnroll; ++u) {
    const int64_t i = lane + 32 * u;
    if (i < nvec) v[u] = ld_stream(xv + i);
  }
  const float L = dbg::ld(lse + row);
  const float L2 = L * kLog2e;
  float gT = dbg::ld(g + row) * invT;
  float pl = 0.f;
  bool bad = false;
  for (int k = lane; k < K; k += 32) {
    const int id = dbg::ld(ids + row * K + k);
    float p = 0.f;
    if (id < 0 || static_cast<int64_t>(id) >= V) {
      bad = true;
      sid[k] = -1;
    } else {
      const float ls = fmaf(E::load1(xr + id), invT, -L);
      p = ls >= clamp_min ? expf(dbg::ld(lt + row * K + k)) : 0.f;
      sid[k] = id;
    }
    sp[k] = p;
    pl += p;
  }
  const float P = warp_sum(pl);  // every lane holds the same sum
  if (__any_sync(0xFFFFFFFFu, bad)) {
    if (lane == 0 && err != nullptr) atomicOr(err, SLP_DATA_ERR_TARGET);
    gT = __int_as_float(0x7FC00000);
  }
  const float dense = gT * P;

  // pass 1: the dense part g/T P q[v] for every element
  const Elt* tag = nullptr;
  const float2 cc = make_float2(c, c);
  const float no1 = log2f(fabsf(dense)) - L2;
  const float2 no = make_float2(no1, no1);
  const uint32_t sgn = sign_mask(dense, tag);
  for (int64_t i0 = lane; i0 < nvec; i0 += 32 * kTkRowsUnroll) {
    if (i0 > lane) {
#pragma unroll
      for (int u = 0; u < kTkRowsUnroll; ++u) {
        const int64_t i = i0 + 32 * u;
        if (i < nvec) v[u] = ld_stream(xv + i);
      }
    }
#pragma unroll
    for (int u = 0; u < kTkRowsUnroll; ++u) {
      const int64_t i = i0 + 32 * u;
      if (i < nvec) st_stream(gv + i, scaled_exp2_vec(v[u], cc, no, sgn, tag));
    }
  }
  for (int64_t e = nvec * kVec + lane; e < V; e += 32)
    E::store1(gr + e, dense * ex2(fmaf(E::load1(xr + e), c, -L2)));

  // pass 2 as in the CTA kernel; the fence and the warp barrier order every
  // lane's pass-1 stores before the rewrites, and make the table visible
  __threadfence_block();
  __syncwarp();
  const int4* sid4 = reinterpret_cast<const int4*>(sid);
  for (int k = lane; k < K; k += 32) {
    const int id = sid[k];
    if (id < 0) continue;
    bool first = true;
    float tot = 0.f;
    for (int j4 = 0; j4 < K4 / 4; ++j4) {
      const int4 q = sid4[j4];
      if (q.x == id || q.y == id || q.z == id || q.w == id) {  // the entry itself, or a repeat
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * j4 + jj;
          if (sid[j] == id) {
            if (j < k) first = false;
            tot += sp[j];
          }
        }
      }
    }
    if (first) {
      const float q = ex2(fmaf(E::load1(xr + id), c, -L2));
      E::store1(gr + id, gT * fmaf(P, q, -tot));
    }
  }
}

bool aligned16(const void* p, int64_t ld, int esize) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ((ld * esize) & 15) == 0;
}

// Measured (bf16, N = 32768, warp per row against CTA per row): 2 KB rows
// 39 against 261 us, 8 KB 120 / 344 us, 16 KB 265 / 439 us, 32 KB 507 /
// 517 us; 64 KB rows 906 / 722 us.
constexpr bool use_topk_rows_kernel(int64_t row_bytes) { return row_bytes <= 32 * 1024; }

template <typename Elt>
cudaError_t topk_bwd_typed(const Elt* x, int64_t N, int64_t V, int64_t ld, const int32_t* ids,
                           const float* lt, int K, const uint8_t* mask, float T, float clamp_min,
                           const float* lse, const float* g, Elt* gx, int64_t ldg, int32_t* err,
                           cudaStream_t stream) {
  const int64_t tables = static_cast<int64_t>(K) * 8;
  if (tables > kTkMaxSmem || N > 0x7FFFFFFFLL) return cudaErrorNotSupported;
  const float invT = 1.0f / T;
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  const bool vec = aligned16(x, ld, sizeof(Elt)) && aligned16(gx, ldg, sizeof(Elt));
  if (vec && K <= kTkRowsMaxK && use_topk_rows_kernel(V * static_cast<int64_t>(sizeof(Elt)))) {
    const int64_t blocks = (N + kTkRowsWarps - 1) / kTkRowsWarps;
    const size_t smem = static_cast<size_t>(kTkRowsWarps) * ((K + 3) & ~3) * 8;
    slp_topk_kl_bwd_rows_kernel<Elt><<<static_cast<unsigned>(blocks), 32 * kTkRowsWarps, smem,
                                       stream>>>(x, N, V, ld, ids, lt, K, mask, invT, c,
                                                 clamp_min, lse, g, gx, ldg, err
                                                 SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, sizeof(Elt)), {ids, 4ull * N * K},
                                  {lt, 4ull * N * K}, {mask, 1ull * N}, {lse, 4ull * N},
                                  {g, 4ull * N}, dbg::rows(gx, N, V, ldg, sizeof(Elt))}));
    return cudaGetLastError();
  }
  auto k = vec ? slp_topk_kl_bwd_kernel<Elt, true> : slp_topk_kl_bwd_kernel<Elt, false>;
  const int64_t smem = vec ? tables + kTkRing : tables;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kTkMaxSmem + kTkRing);
  if (e != cudaSuccess) return e;
  k<<<static_cast<unsigned>(N), kTkThreads, static_cast<size_t>(smem), stream>>>(
      x, V, ld, ids, lt, K, mask, invT, c, clamp_min, lse, g, gx, ldg, err
      SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, sizeof(Elt)), {ids, 4ull * N * K},
                                  {lt, 4ull * N * K}, {mask, 1ull * N}, {lse, 4ull * N},
                                  {g, 4ull * N}, dbg::rows(gx, N, V, ldg, sizeof(Elt))}));
  return cudaGetLastError();
}

}  // namespace

int64_t topk_kl_max_k() { return kTkMaxSmem / 8; }

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
        mask, invT, clamp_min, lse, kl, student_mass, teacher_mass, err
        SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, 2), {ids, 4ull * N * K},
                          {teacher_logp, 4ull * N * K}, {mask, 1ull * N}, {lse, 4ull * N},
                          {kl, 4ull * N}, {student_mass, 4ull * N}, {teacher_mass, 4ull * N}}));
  else
    slp_topk_kl_rows_kernel<float><<<blocks, 256, 0, stream>>>(
        static_cast<const float*>(x), N, V, ld, ids, teacher_logp, static_cast<int>(K), mask,
        invT, clamp_min, lse, kl, student_mass, teacher_mass, err
        SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, 4), {ids, 4ull * N * K},
                          {teacher_logp, 4ull * N * K}, {mask, 1ull * N}, {lse, 4ull * N},
                          {kl, 4ull * N}, {student_mass, 4ull * N}, {teacher_mass, 4ull * N}}));
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
