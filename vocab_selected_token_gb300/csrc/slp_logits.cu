// Logits-input path: forward (online log-sum-exp + target gather) and
// backward ((onehot - softmax) * g / T with the softmax recomputed from the
// saved lse), both streaming kernels bound by HBM bandwidth.
//
// Forward: one CTA per row (a thread-block cluster of `splits` CTAs per row
// when there are too few rows to fill the GPU).  For 16-byte-aligned rows,
// thread 0 streams the row segment into a 4 x 16 KB shared-memory ring with
// cp.async.bulk copies completing on mbarriers, so ~64 KB per CTA is always
// in flight while all 256 threads fold the landed chunks into a running
// base-2 (max, sum-exp) state.  Warps merge by butterfly shuffles, CTAs of a
// cluster through distributed shared memory: the single-GPU form of the
// vocabulary-parallel exchange (torchforge PR #608, "Implementation":
// all-reduce MAX, all-reduce SUM of exp(x - max), target gathered by its
// owner only), with no global workspace.
//
// Backward: a flat grid of (row, column-tile) CTAs; each thread handles
// kBwdUnroll 16-byte vectors, recomputes p = 2^(x*c - lse*log2 e) and writes
// g/T * (1[v == t] - p) with streaming stores.  Inactive rows only write zeros.
//
// Fused forward + backward (the upstream gradient known at forward time): a
// cluster of CTAs holds each row on chip between the two passes (registers,
// shared memory and, for long fp32 rows, tensor memory), so the row is read
// from HBM once.
//
// Short rows (a few KB, small vocabularies) take kernels with one warp per
// row instead, for the forward, the backward and the fused call: one CTA per
// row spends more on its set-up than on such a row's traffic.

#include "slp.h"
#include "slp_device.cuh"
#include "slp_internal.h"
#include "slp_sm100.cuh"

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <type_traits>

namespace slp {

constexpr int kFwdThreads = 256;
constexpr int kFwdChunk = 16384;  // bytes per bulk copy (4 vectors per thread)
// Shared-memory ring of the vector path, in chunks: four (64 KB, three CTAs
// per SM) for the plain log-sum-exp; two (32 KB, six CTAs per SM) with the
// entropy accumulator, whose fold has more arithmetic per byte and gains more
// from extra warps than from a deeper ring (measured: 0.196 -> 0.183 ms on
// c151k; the plain fold is the same with three or four stages).
template <typename St>
__host__ __device__ constexpr int fwd_stages() { return sizeof(St) == sizeof(Lse3) ? 2 : 4; }
template <typename St>
__host__ __device__ constexpr int fwd_smem() { return fwd_stages<St>() * kFwdChunk; }
constexpr uint64_t kFwdWaitNs = 2000000000ull;
constexpr int kBwdThreads = 256;
constexpr int kBwdUnroll = 4;
constexpr int kMaxSplits = 8;  // portable cluster size

// St is Lse2 (log-prob and lse) or Lse3 (also the entropy, written to
// `entropy`, which is otherwise unused).
template <typename Elt, bool kVecPath, typename St>
__global__ void __launch_bounds__(kFwdThreads)
    slp_fwd_kernel(const Elt* __restrict__ x, int64_t V, int64_t ld,
                   const int32_t* __restrict__ t, const uint8_t* __restrict__ mask, float T,
                   float c, float* __restrict__ logprob, float* __restrict__ lse,
                   float* __restrict__ entropy, int32_t* __restrict__ err, int splits SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  using E = Elem<Elt>;
  constexpr int kVec = E::kVec;
  constexpr int kWarps = kFwdThreads / 32;
  constexpr bool kEnt = sizeof(St) == sizeof(Lse3);
  constexpr int kFwdStages = fwd_stages<St>();
  __shared__ St warp_part[kWarps];
  __shared__ float cta_part[4];

  const int64_t row = blockIdx.x / splits;
  const int rank = static_cast<int>(blockIdx.x - row * splits);
  // Every CTA of a cluster handles the same row, so all of them leave here
  // together (no cluster barrier is left waiting).
  if (mask != nullptr && dbg::ld(mask + row) == 0) {
    if (rank == 0 && threadIdx.x == 0) {
      if (logprob != nullptr) dbg::st(logprob + row, 0.f);
      dbg::st(lse + row, 0.f);
      if (kEnt) dbg::st(entropy + row, 0.f);
    }
    return;
  }
  const Elt* xr = x + row * ld;
  // t == NULL: log-sum-exp only (no target, logprob not written)
  const int32_t tt = t != nullptr ? dbg::ld(t + row) : 0;
  const bool tvalid = tt >= 0 && static_cast<int64_t>(tt) < V;
  float xt = 0.f;
  if (rank == 0 && threadIdx.x == 0 && tvalid) xt = E::load1(xr + tt);

  St st;
  st_empty(st);
  if constexpr (kVecPath) {
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t full[kFwdStages];
    __shared__ int abort_flag;
    const int64_t nvec = V / kVec;
    const int64_t v0 = nvec * rank / splits;
    const int64_t v1 = nvec * (rank + 1) / splits;
    const char* src = reinterpret_cast<const char*>(reinterpret_cast<const uint4*>(xr) + v0);
    const int64_t nbytes = (v1 - v0) * 16;
    const int64_t nch = (nbytes + kFwdChunk - 1) / kFwdChunk;
    const uint32_t sbase = sm100::smem_u32(ring);
    const uint32_t bbase = sm100::smem_u32(full);
    if (threadIdx.x == 0) {
      for (int s = 0; s < kFwdStages; ++s) sm100::mbar_init(bbase + 8 * s, 1);
      abort_flag = 0;
      sm100::fence_mbar_init();
    }
    __syncthreads();
    // thread 0 keeps kFwdStages chunks of the segment in flight
    auto issue = [&](int64_t ch) {
      const int s = static_cast<int>(ch % kFwdStages);
      const int64_t off = ch * kFwdChunk;
      const uint32_t bytes = static_cast<uint32_t>(
          nbytes - off < kFwdChunk ? nbytes - off : static_cast<int64_t>(kFwdChunk));
      sm100::mbar_arrive_expect_tx(bbase + 8 * s, bytes);
      sm100::bulk_load(sbase + s * kFwdChunk, src + off, bytes, bbase + 8 * s);
    };
    if (threadIdx.x == 0)
      for (int64_t ch = 0; ch < kFwdStages && ch < nch; ++ch) issue(ch);
    constexpr int kPer = kFwdChunk / 16 / kFwdThreads;
    const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
    int64_t ch = 0;
    for (; ch < nch; ++ch) {
      const int s = static_cast<int>(ch % kFwdStages);
      const bool got = sm100::mbar_wait_bounded(bbase + 8 * s, (ch / kFwdStages) & 1,
                                                &abort_flag, kFwdWaitNs);
      if (__syncthreads_or(!got)) break;
      const int64_t off = ch * kFwdChunk;
      const int nv = static_cast<int>(
          (nbytes - off < kFwdChunk ? nbytes - off : static_cast<int64_t>(kFwdChunk)) / 16);
      const uint4* q = reinterpret_cast<const uint4*>(ring + s * kFwdChunk);
      uint4 vv[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = u * kFwdThreads + threadIdx.x;
        vv[u] = i < nv ? q[i] : pad;
      }
      sm100::fence_proxy_async_smem();  // these reads precede the refill below
      __syncthreads();  // stage s fully read: thread 0 may refill it
      if (threadIdx.x == 0 && ch + kFwdStages < nch) issue(ch + kFwdStages);
      if constexpr (kEnt)
        lse3_fold_vec<kPer>(st, vv, c, static_cast<const Elt*>(nullptr));
      else
        lse2_fold_vec<kPer>(st, vv, c, static_cast<const Elt*>(nullptr));
    }
    if (ch < nch) {
      // a copy never landed: report it and wait (bounded) for the copies in
      // flight so the CTA does not exit under them
      if (threadIdx.x == 0) {
        if (err != nullptr) atomicOr(err, SLP_DEVICE_ERR_TIMEOUT);
        const int64_t last = (ch + kFwdStages < nch ? ch + kFwdStages : nch);
        for (int64_t j = ch; j < last; ++j)
          sm100::mbar_wait_bounded(bbase + 8 * (j % kFwdStages), (j / kFwdStages) & 1, nullptr,
                                   kFwdWaitNs);
      }
      __syncthreads();
    }
    if (rank == splits - 1) {  // fewer than kVec trailing elements
      const int64_t e = nvec * kVec + threadIdx.x;
      if (e < V) {
        float f1[1] = {E::load1(xr + e)};
        st_fold<1>(st, f1, c);
      }
    }
  } else {
    const int64_t e0 = V * rank / splits;
    const int64_t e1 = V * (rank + 1) / splits;
    for (int64_t i0 = e0 + threadIdx.x; i0 < e1; i0 += kFwdThreads * 4) {
      float f[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i = i0 + static_cast<int64_t>(u) * kFwdThreads;
        f[u] = (i < e1) ? E::load1(xr + i) : -INFINITY;
      }
      st_fold<4>(st, f, c);
    }
  }

  // CTA merge: warps, then the warp results in warp order.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  st = st_warp_reduce(st);
  if (lane == 0) warp_part[warp] = st;
  __syncthreads();
  auto finish = [&](const St& v) {
    if constexpr (kEnt)
      write_row_result(v, xt, tvalid, T, c, logprob, lse, entropy, err, row);
    else
      write_row_result(v, xt, tvalid, T, c, logprob, lse, err, row);
  };
  if (warp == 0) {
    St v;
    if (lane < kWarps) v = warp_part[lane];
    else st_empty(v);
    v = st_warp_reduce(v);
    if (lane == 0) {
      const float* vf = reinterpret_cast<const float*>(&v);
#pragma unroll
      for (int k = 0; k < static_cast<int>(sizeof(St) / 4); ++k) cta_part[k] = vf[k];
      if (splits == 1) finish(v);
    }
  }
  if (splits == 1) return;

  // Cluster merge: in CTA rank 0, lane r of warp 0 reads rank r's state over
  // DSMEM (the reads overlap) and lane 0 merges them in rank order.  Only
  // thread 0 of each CTA wrote its state, so only it fences before the
  // barrier.  The second barrier keeps every CTA resident until those reads
  // are done.
  constexpr int kF = static_cast<int>(sizeof(St) / 4);
  cluster_sync_from_thread0();
  if (rank == 0 && warp == 0) {
    St o;
    st_empty(o);
    float* of = reinterpret_cast<float*>(&o);
    if (lane < splits) {
#pragma unroll
      for (int k = 0; k < kF; ++k) of[k] = ld_shared_cluster_f32(map_shared_rank(&cta_part[k], lane));
    }
    St acc;
    st_empty(acc);
    for (int r = 0; r < splits; ++r) {
      St pr;
      float* pf = reinterpret_cast<float*>(&pr);
#pragma unroll
      for (int k = 0; k < kF; ++k) pf[k] = __shfl_sync(0xFFFFFFFFu, of[k], r);
      acc = st_merge(acc, pr);
    }
    if (lane == 0) finish(acc);
  }
  asm volatile("barrier.cluster.arrive.relaxed;\n\t"
               "barrier.cluster.wait.acquire;" ::
                   : "memory");
}

// Short rows: one warp per row, eight rows per CTA, plain 16-byte streaming
// loads kRowsUnroll deep per lane and no shared memory or CTA barrier.  For
// such rows the per-CTA set-up of the ring kernel (one CTA per row) costs more
// than the row's own traffic.  Same fold and same row result as the ring
// kernel.  Measured against it (forward, bf16, TB/s): V = 8192, N = 4096:
// 5.33 against 2.16; V = 32768, N = 16384: 6.68 against 5.12; at V = 65536
// the two tie, and above it, or for few rows, the ring kernel is ahead.
constexpr int kRowsWarps = 8;
constexpr int kRowsUnroll = 8;

__host__ __device__ constexpr bool use_rows_kernel(int64_t N, int64_t row_bytes) {
  return row_bytes <= 32 * 1024 || (row_bytes <= 64 * 1024 && N >= 2048);
}

template <typename Elt, typename St>
__global__ void __launch_bounds__(32 * kRowsWarps)
    slp_fwd_rows_kernel(const Elt* __restrict__ x, int64_t N, int64_t V, int64_t ld,
                        const int32_t* __restrict__ t, const uint8_t* __restrict__ mask, float T,
                        float c, float* __restrict__ logprob, float* __restrict__ lse,
                        float* __restrict__ entropy, int32_t* __restrict__ err SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  using E = Elem<Elt>;
  constexpr int kVec = E::kVec;
  constexpr bool kEnt = sizeof(St) == sizeof(Lse3);
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsWarps + (threadIdx.x >> 5);
  if (row >= N) return;
  if (mask != nullptr && dbg::ld(mask + row) == 0) {
    if (lane == 0) {
      if (logprob != nullptr) dbg::st(logprob + row, 0.f);
      dbg::st(lse + row, 0.f);
      if (kEnt) dbg::st(entropy + row, 0.f);
    }
    return;
  }
  const Elt* xr = x + row * ld;
  const uint4* xv = reinterpret_cast<const uint4*>(xr);
  const int64_t nvec = V / kVec;
  const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
  St st;
  st_empty(st);
  for (int64_t i0 = lane; i0 < nvec; i0 += 32 * kRowsUnroll) {
    uint4 v[kRowsUnroll];
#pragma unroll
    for (int u = 0; u < kRowsUnroll; ++u) {
      const int64_t i = i0 + 32 * u;
      v[u] = i < nvec ? ld_stream(xv + i) : pad;
    }
    if constexpr (kEnt)
      lse3_fold_vec<kRowsUnroll>(st, v, c, static_cast<const Elt*>(nullptr));
    else
      lse2_fold_vec<kRowsUnroll>(st, v, c, static_cast<const Elt*>(nullptr));
  }
  for (int64_t e = nvec * kVec + lane; e < V; e += 32) {  // fewer than kVec trailing elements
    float f1[1] = {E::load1(xr + e)};
    st_fold<1>(st, f1, c);
  }
  st = st_warp_reduce(st);
  if (lane == 0) {
    const int32_t tt = t != nullptr ? dbg::ld(t + row) : 0;
    const bool tvalid = tt >= 0 && static_cast<int64_t>(tt) < V;
    const float xt = tvalid ? E::load1(xr + tt) : 0.f;
    if constexpr (kEnt)
      write_row_result(st, xt, tvalid, T, c, logprob, lse, entropy, err, row);
    else
      write_row_result(st, xt, tvalid, T, c, logprob, lse, err, row);
  }
}

// Per-row terms of the backward.  Off the target an element's gradient is
// a p with a = -g/T, or with the entropy term (kEnt; H and gH per row, g and
// gH may then be NULL, meaning zero) p (a - gH/T ln 2 (log2 p + H log2 e)) =
// p (a2 + gHl log2 p); the target's element adds g/T.  vec() does a 16-byte
// vector of off-target elements in paired arithmetic (scaled_exp2_vec /
// entropy_grad_vec), one() a single element in full.  log2 p is clamped at
// -256 with the entropy term, so a -inf logit gives p = 0 and a finite
// factor.
template <typename Elt, bool kEnt>
struct BwdRow {
  float gT, L2, Hl2, gHl, a;
  int64_t tt;
  float2 cc, no, gHl2, a2;
  uint32_t sgn;

  // report: this thread flags a bad target in *err (one thread per row)
  __device__ __forceinline__ void init(int64_t row, int64_t V, const int32_t* t, float invT,
                                       float c, const float* lse, const float* g, const float* H,
                                       const float* gH, int32_t* err, bool report) {
    const Elt* tag = nullptr;
    tt = dbg::ld(t + row);
    gT = (kEnt && g == nullptr) ? 0.f : dbg::ld(g + row) * invT;
    L2 = dbg::ld(lse + row) * kLog2e;
    float gHT = 0.f;
    Hl2 = 0.f;
    if (kEnt) {
      gHT = gH == nullptr ? 0.f : dbg::ld(gH + row) * invT;
      Hl2 = dbg::ld(H + row) * kLog2e;  // log p_v + H = ln 2 (log2 p_v + H log2 e)
    }
    if (tt < 0 || tt >= V) {
      if (err != nullptr && report) atomicOr(err, SLP_DATA_ERR_TARGET);
      gT = __int_as_float(0x7FC00000);
    }
    a = -gT;
    gHl = -gHT * kLn2;
    cc = make_float2(c, c);
    const float no1 = kEnt ? -L2 : log2f(fabsf(a)) - L2;  // -(L2 - log2 |a|) without entropy
    no = make_float2(no1, no1);
    sgn = sign_mask(a, tag);
    gHl2 = make_float2(gHl, gHl);
    const float a2s = fmaf(gHl, Hl2, a);
    a2 = make_float2(a2s, a2s);
  }
  // The same terms from values already in registers (the fused kernels):
  // gT0 = g/T (NaN for a bad target), L20 = lse log2 e, gHT = gH/T,
  // Hl20 = H log2 e.  The derived terms repeat init's lines: routing init
  // through this function instead changed the plain backward's schedule and
  // cost it 2.5 % (353 -> 362 us on c151k).
  __device__ __forceinline__ void set(int64_t t0, float gT0, float L20, float gHT, float Hl20,
                                      float c) {
    const Elt* tag = nullptr;
    tt = t0;
    gT = gT0;
    L2 = L20;
    Hl2 = kEnt ? Hl20 : 0.f;
    a = -gT;
    gHl = -gHT * kLn2;
    cc = make_float2(c, c);
    const float no1 = kEnt ? -L2 : log2f(fabsf(a)) - L2;
    no = make_float2(no1, no1);
    sgn = sign_mask(a, tag);
    gHl2 = make_float2(gHl, gHl);
    const float a2s = fmaf(gHl, Hl2, a);
    a2 = make_float2(a2s, a2s);
  }
  __device__ __forceinline__ uint4 vec(const uint4& v) const {
    const Elt* tag = nullptr;
    return kEnt ? entropy_grad_vec(v, cc, no, gHl2, a2, tag) : scaled_exp2_vec(v, cc, no, sgn, tag);
  }
  __device__ __forceinline__ float one(float x, float c, bool is_t) const {
    float l2p = fmaf(x, c, -L2);
    if (kEnt) l2p = fmaxf(l2p, -256.f);
    const float p = ex2(l2p);
    const float w = kEnt ? fmaf(gHl, l2p + Hl2, a) : a;
    return is_t ? fmaf(w, p, gT) : w * p;
  }
};

// With the entropy term the register count would leave three or four CTAs
// per SM; capping it for six measured 0.375 -> 0.360 ms on c151k.
template <typename Elt, bool kVecPath, bool kEnt>
__global__ void __launch_bounds__(kBwdThreads, kEnt ? 6 : 1)
    slp_bwd_kernel(const Elt* __restrict__ x, int64_t V, int64_t ld,
                   const int32_t* __restrict__ t, const uint8_t* __restrict__ mask, float invT,
                   float c, const float* __restrict__ lse, const float* __restrict__ g,
                   const float* __restrict__ H, const float* __restrict__ gH,
                   Elt* __restrict__ gx, int64_t ldg, int32_t* __restrict__ err,
                   int64_t tiles_per_row SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  using E = Elem<Elt>;
  constexpr int kVec = E::kVec;
  constexpr int64_t kTileElems = static_cast<int64_t>(kBwdThreads) * kBwdUnroll * kVec;

  const int64_t row = blockIdx.x / tiles_per_row;
  const int64_t tile = blockIdx.x - row * tiles_per_row;
  const bool active = mask == nullptr || dbg::ld(mask + row) != 0;
  const Elt* xr = x + row * ld;
  Elt* gr = gx + row * ldg;
  const int64_t e_tile = tile * kTileElems;
  BwdRow<Elt, kEnt> b;
  if (active) b.init(row, V, t, invT, c, lse, g, H, gH, err, tile == 0 && threadIdx.x == 0);

  if constexpr (kVecPath) {
    uint4* gv = reinterpret_cast<uint4*>(gr);
    const uint4* xv = reinterpret_cast<const uint4*>(xr);
    if (!active) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < kBwdUnroll; ++u) {
        const int64_t e = e_tile + (static_cast<int64_t>(u) * kBwdThreads + threadIdx.x) * kVec;
        if (e + kVec <= V) {
          st_stream(gv + e / kVec, z);
        } else {
          for (int64_t k = e; k < V; ++k) E::store1(gr + k, 0.f);
        }
      }
      return;
    }
    uint4 buf[kBwdUnroll];
#pragma unroll
    for (int u = 0; u < kBwdUnroll; ++u) {
      const int64_t e = e_tile + (static_cast<int64_t>(u) * kBwdThreads + threadIdx.x) * kVec;
      if (e + kVec <= V) buf[u] = ld_stream(xv + e / kVec);
    }
    // The thread whose vector holds the target stores that element again, in
    // full, after the vector (same thread: it lands last).
#pragma unroll
    for (int u = 0; u < kBwdUnroll; ++u) {
      const int64_t e = e_tile + (static_cast<int64_t>(u) * kBwdThreads + threadIdx.x) * kVec;
      if (e + kVec <= V) {
        st_stream(gv + e / kVec, b.vec(buf[u]));
        if (b.tt >= e && b.tt < e + kVec) E::store1(gr + b.tt, b.one(E::load1(xr + b.tt), c, true));
      } else {
        for (int64_t k = e; k < V; ++k) E::store1(gr + k, b.one(E::load1(xr + k), c, k == b.tt));
      }
    }
  } else {
    const int64_t e_end = min(V, e_tile + kTileElems);
    for (int64_t e = e_tile + threadIdx.x; e < e_end; e += kBwdThreads)
      E::store1(gr + e, active ? b.one(E::load1(xr + e), c, e == b.tt) : 0.f);
  }
}

// Short rows: the backward with one warp per row (the grid above gives each
// row tiles of 8192 elements, which a short row leaves mostly idle).  Same
// per-element arithmetic as slp_bwd_kernel, so the same bits.
template <typename Elt, bool kEnt>
__global__ void __launch_bounds__(32 * kRowsWarps)
    slp_bwd_rows_kernel(const Elt* __restrict__ x, int64_t N, int64_t V, int64_t ld,
                        const int32_t* __restrict__ t, const uint8_t* __restrict__ mask,
                        float invT, float c, const float* __restrict__ lse,
                        const float* __restrict__ g, const float* __restrict__ H,
                        const float* __restrict__ gH, Elt* __restrict__ gx, int64_t ldg,
                        int32_t* __restrict__ err SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  using E = Elem<Elt>;
  constexpr int kVec = E::kVec;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsWarps + (threadIdx.x >> 5);
  if (row >= N) return;
  const int64_t nvec = V / kVec;
  Elt* gr = gx + row * ldg;
  uint4* gv = reinterpret_cast<uint4*>(gr);
  if (mask != nullptr && dbg::ld(mask + row) == 0) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t i = lane; i < nvec; i += 32) st_stream(gv + i, z);
    for (int64_t e = nvec * kVec + lane; e < V; e += 32) E::store1(gr + e, 0.f);
    return;
  }
  const Elt* xr = x + row * ld;
  const uint4* xv = reinterpret_cast<const uint4*>(xr);
  BwdRow<Elt, kEnt> b;
  b.init(row, V, t, invT, c, lse, g, H, gH, err, lane == 0);
  for (int64_t i0 = lane; i0 < nvec; i0 += 32 * kRowsUnroll) {
    uint4 v[kRowsUnroll];
#pragma unroll
    for (int u = 0; u < kRowsUnroll; ++u) {
      const int64_t i = i0 + 32 * u;
      if (i < nvec) v[u] = ld_stream(xv + i);
    }
#pragma unroll
    for (int u = 0; u < kRowsUnroll; ++u) {
      const int64_t i = i0 + 32 * u;
      if (i < nvec) {
        st_stream(gv + i, b.vec(v[u]));
        const int64_t e = i * kVec;
        if (b.tt >= e && b.tt < e + kVec) E::store1(gr + b.tt, b.one(E::load1(xr + b.tt), c, true));
      }
    }
  }
  for (int64_t e = nvec * kVec + lane; e < V; e += 32)  // fewer than kVec trailing elements
    E::store1(gr + e, b.one(E::load1(xr + e), c, e == b.tt));
}


// ---- fused forward + backward (upstream gradient known at forward time) ----
//
// A cluster of C CTAs holds one row on chip, each CTA a contiguous segment:
// its last kFbRV vectors per thread in registers (plain 16-byte loads), the
// rest in shared memory (bulk copies).  Holding part of the row in registers
// lets four CTAs share an SM instead of three, so more rows are in flight
// while each row's CTAs wait for one another.  The log-sum-exp is folded as
// the data lands and merged across the cluster through distributed shared
// memory: every CTA merges all partials in rank order, so all of them hold
// the same state.  Each CTA then writes its segment of
// g/T * (1[v == t] - p) straight from registers and shared memory.  That is one
// HBM read of the active rows plus one write of the gradient, instead of the
// two reads of a separate forward and backward (NeMo-RL PR #4222, "Changes":
// recompute the softmax instead of storing it; here the row stays on chip
// between the two passes).  The row is read with an L2 evict-first policy:
// it is read once, and L2 is better left to the gradient's write-back
// (measured on c151k: 402 -> 394 us).  Long fp32 rows also keep kFbTV more
// vectors per thread in tensor memory (the TMEM part, see tmem_fused_form),
// so their clusters need fewer CTAs.

constexpr int kFbThreads = 256;
constexpr int kFbChunk = 16384;
// Register part: kFbRV 16-byte vectors per thread.  With at most 64 registers
// per thread and kFbMaxSmem bytes of shared memory, four CTAs stay resident
// per SM (228 KB of shared memory per SM, less 1 KB reserved and 256 B static
// per CTA); kFbRegSeg is the segment that fits.
constexpr int kFbMaxSmem = 233472 / 4 - 1024 - 256;
constexpr int kFbMaxChunks = (kFbMaxSmem + kFbChunk - 1) / kFbChunk;
constexpr int kFbRV = 5;
constexpr int kFbRegSeg = kFbMaxSmem + kFbRV * kFbThreads * 16;
constexpr int kFbMaxCluster = 8;
// TMEM part: kFbTV more vectors per thread in tensor memory (tcgen05.st /
// tcgen05.ld, 32 lanes x 4 kFbTV columns per warp, 128 columns per CTA).  An
// SM's 512 TMEM columns hold four such CTAs, so the form reserves at least
// kFbTmMinSmem bytes of shared memory per CTA: a fifth CTA never fits on an
// SM, and no tcgen05.alloc ever waits for columns.
constexpr int kFbTV = 16;
constexpr int kFbTmCols = 128;
constexpr int kFbTmMinSmem = 233472 / 5 - 1024 - 256 + 1;  // 5 CTAs would need more
constexpr int kFbTmSeg = kFbRegSeg + kFbTV * kFbThreads * 16;

// The TMEM part in pass 2: kTV vectors of this thread read back four at a
// time (16 columns per tcgen05.ld), each handed to put(i, v).
template <int kTV, typename Put>
__device__ __forceinline__ void put_tmem(uint32_t taddr, int nv_s, int nv, Put& put) {
#pragma unroll 1
  for (int b = 0; b < kTV / 4; ++b) {
    uint4 tv[4];
    sm100::tmem_ld_4vec(taddr + 16 * b, tv);
    sm100::tmem_ld_wait();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = nv_s + (4 * b + u) * kFbThreads + threadIdx.x;
      if (i < nv) put(i, tv[u]);
    }
  }
}

// Every thread has finished with TMEM: warp 0 frees the CTA's columns.
__device__ __forceinline__ void free_tmem(uint32_t base) {
  sm100::tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    sm100::tc_fence_after();
    sm100::tmem_dealloc(base, kFbTmCols);
  }
}

// kEnt adds the entropy: the state carries the entropy accumulator, the row
// results include H (`entropy`), and the gradient gains the entropy term
// -gH p (log p + H) / T computed from the lse and H written here, exactly as
// slp_bwd_kernel computes it from the saved ones (g and gH may then be NULL,
// meaning zero).
template <typename Elt, int kTV, bool kEnt>
__global__ void __launch_bounds__(kFbThreads, 4)
    slp_fwd_bwd_kernel(const Elt* __restrict__ x, int64_t V, int64_t ld,
                       const int32_t* __restrict__ t, const uint8_t* __restrict__ mask, float T,
                       float c, float invT, const float* __restrict__ g,
                       const float* __restrict__ gH, float* __restrict__ logprob,
                       float* __restrict__ lse, float* __restrict__ entropy,
                       Elt* __restrict__ gx, int64_t ldg, int32_t* __restrict__ err, int C SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  using E = Elem<Elt>;
  using St = typename std::conditional<kEnt, Lse3, Lse2>::type;
  constexpr int kVec = E::kVec;
  constexpr int kWarps = kFbThreads / 32;
  extern __shared__ __align__(128) uint8_t seg[];
  __shared__ __align__(8) uint64_t full[kFbMaxChunks];
  __shared__ St warp_part[kWarps];
  __shared__ float cta_part[4];
  __shared__ int abort_flag;

  const int64_t row = blockIdx.x / C;
  const int rank = static_cast<int>(blockIdx.x - row * C);
  const int64_t nvec = V / kVec;
  const int64_t v0 = nvec * rank / C;
  const int64_t v1 = nvec * (rank + 1) / C;
  const int nv = static_cast<int>(v1 - v0);  // vectors of this segment
  // the last kRV * kFbThreads vectors of the segment stay in registers (kRV
  // per thread), the kTV * kFbThreads before them in TMEM (kTV per thread),
  // the rest in shared memory
  constexpr int kRV = kFbRV;
  constexpr int kRegVec = kRV * kFbThreads;
  constexpr int kTmVec = kTV * kFbThreads;
  const int nv_s = nv > kRegVec + kTmVec ? nv - kRegVec - kTmVec : 0;
  const int nv_r = nv_s + kTmVec;  // first vector of the register part
  const Elt* tag = nullptr;
  uint4* gv = reinterpret_cast<uint4*>(gx + row * ldg) + v0;

  // Inactive rows: every CTA of the cluster writes zeros and leaves; none of
  // them touches a cluster barrier.
  if (mask != nullptr && dbg::ld(mask + row) == 0) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < nv; i += kFbThreads) st_stream(gv + i, z);
    if (rank == C - 1)
      for (int64_t e = nvec * kVec + threadIdx.x; e < V; e += kFbThreads)
        E::store1(gx + row * ldg + e, 0.f);
    if (rank == 0 && threadIdx.x == 0) {
      dbg::st(logprob + row, 0.f);
      dbg::st(lse + row, 0.f);
      if (kEnt) dbg::st(entropy + row, 0.f);
    }
    return;
  }

  const Elt* xr = x + row * ld;
  const int32_t tt = dbg::ld(t + row);
  const bool tvalid = tt >= 0 && static_cast<int64_t>(tt) < V;
  float xt = 0.f;
  if (rank == 0 && threadIdx.x == 0 && tvalid) xt = E::load1(xr + tt);
  const float gT = tvalid ? ((kEnt && g == nullptr) ? 0.f : dbg::ld(g + row) * invT)
                          : __int_as_float(0x7FC00000);

  const int seg_bytes = nv_s * 16;
  const int nch = (seg_bytes + kFbChunk - 1) / kFbChunk;
  const uint32_t sbase = sm100::smem_u32(seg);
  const uint32_t bbase = sm100::smem_u32(full);
  if (threadIdx.x == 0) {
    for (int k = 0; k < nch; ++k) sm100::mbar_init(bbase + 8 * k, 1);
    abort_flag = 0;
    sm100::fence_mbar_init();
  }
  __shared__ uint32_t tmem_holder;
  if constexpr (kTV > 0) {
    if (threadIdx.x < 32) sm100::tmem_alloc(sm100::smem_u32(&tmem_holder), kFbTmCols);
    sm100::tc_fence_before();
  }
  __syncthreads();
  uint32_t taddr = 0;  // this thread's TMEM lane and first column
  if constexpr (kTV > 0) {
    sm100::tc_fence_after();
    const int w = threadIdx.x >> 5;
    taddr = tmem_holder + (static_cast<uint32_t>((w & 3) * 32) << 16) +
            static_cast<uint32_t>((w >> 2) * kTV * 4);
  }
  if (threadIdx.x == 0) {
    const char* src = reinterpret_cast<const char*>(reinterpret_cast<const uint4*>(xr) + v0);
    for (int k = 0; k < nch; ++k) {
      const int off = k * kFbChunk;
      const uint32_t bytes = static_cast<uint32_t>(seg_bytes - off < kFbChunk ? seg_bytes - off
                                                                                : kFbChunk);
      sm100::mbar_arrive_expect_tx(bbase + 8 * k, bytes);
      sm100::bulk_load_ef(sbase + off, src + off, bytes, bbase + 8 * k);
    }
  }

  const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
  uint4 rv[kRV];  // the register part, loaded while the chunks stream in
  {
    const uint4* xv = reinterpret_cast<const uint4*>(xr) + v0;
#pragma unroll
    for (int u = 0; u < kRV; ++u) {
      const int i = nv_r + u * kFbThreads + threadIdx.x;
      rv[u] = i < nv ? ld_stream_ef(xv + i) : pad;
    }
  }

  // pass 1: online log-sum-exp over the segment as its chunks land
  St st;
  st_empty(st);
  if constexpr (kTV > 0) {
    // TMEM part, four vectors at a time: loaded, folded, stored to this
    // thread's lane (16 columns per tcgen05.st)
    const uint4* xv = reinterpret_cast<const uint4*>(xr) + v0;
    auto load4 = [&](uint4 (&tv)[4], int b) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = nv_s + (4 * b + u) * kFbThreads + threadIdx.x;
        tv[u] = i < nv ? ld_stream_ef(xv + i) : pad;
      }
    };
#pragma unroll 1
    for (int b = 0; b < kTV / 4; ++b) {
      uint4 tv[4];
      load4(tv, b);
      if constexpr (kEnt)
        lse3_fold_vec<4>(st, tv, c, tag);
      else
        lse2_fold_vec<4>(st, tv, c, tag);
      sm100::tmem_st_4vec(taddr + 16 * b, tv);
    }
    sm100::tmem_st_wait();
  }
  const uint4* q = reinterpret_cast<const uint4*>(seg);
  constexpr int kPer = kFbChunk / 16 / kFbThreads;
  bool ok = true;
  for (int k = 0; k < nch; ++k) {
    // each thread waits on its own; one that gives up sets abort_flag, which
    // ends the others' waits, and the CTA agrees on `ok` after the loop
    if (!sm100::mbar_wait_bounded(bbase + 8 * k, 0, &abort_flag, kFwdWaitNs)) {
      ok = false;
      break;
    }
    uint4 vv[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = k * (kFbChunk / 16) + u * kFbThreads + threadIdx.x;
      vv[u] = i < nv_s ? q[i] : pad;
    }
    if constexpr (kEnt)
      lse3_fold_vec<kPer>(st, vv, c, tag);
    else
      lse2_fold_vec<kPer>(st, vv, c, tag);
  }
  ok = !__syncthreads_or(!ok);
  if constexpr (kEnt)
    lse3_fold_vec<kRV>(st, rv, c, tag);
  else
    lse2_fold_vec<kRV>(st, rv, c, tag);
  if (!ok && threadIdx.x == 0) {
    if (err != nullptr) atomicOr(err, SLP_DEVICE_ERR_TIMEOUT);
    for (int k = 0; k < nch; ++k)  // let every copy land before the CTA moves on
      sm100::mbar_wait_bounded(bbase + 8 * k, 0, nullptr, kFwdWaitNs);
  }
  if (rank == C - 1) {
    const int64_t e = nvec * kVec + threadIdx.x;
    if (e < V) {
      float f1[1] = {E::load1(xr + e)};
      st_fold<1>(st, f1, c);
    }
  }

  // CTA merge, then cluster merge (every CTA reads all partials)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  st = st_warp_reduce(st);
  if (lane == 0) warp_part[warp] = st;
  __syncthreads();
  if (warp == 0) {
    St v;
    if (lane < kWarps)
      v = warp_part[lane];
    else
      st_empty(v);
    v = st_warp_reduce(v);
    if (lane == 0) {
      cta_part[0] = v.m;
      cta_part[1] = v.mc;
      cta_part[2] = v.s;
      if constexpr (kEnt) cta_part[3] = v.w;
    }
  }
  cluster_sync_from_thread0();  // thread 0 wrote cta_part
  __shared__ St row_state;
  if (warp == 0) {
    // lane r fetches rank r's partial (the C remote reads overlap), then
    // every lane merges them in rank order
    St o;
    st_empty(o);
    if (lane < C) {
      const uint32_t b = map_shared_rank(&cta_part[0], lane);
      o.m = ld_shared_cluster_f32(b);
      o.mc = ld_shared_cluster_f32(b + 4);
      o.s = ld_shared_cluster_f32(b + 8);
      if constexpr (kEnt) o.w = ld_shared_cluster_f32(b + 12);
    }
    St acc;
    st_empty(acc);
    for (int r = 0; r < C; ++r) {
      St pr;
      pr.m = __shfl_sync(0xFFFFFFFFu, o.m, r);
      pr.mc = __shfl_sync(0xFFFFFFFFu, o.mc, r);
      pr.s = __shfl_sync(0xFFFFFFFFu, o.s, r);
      if constexpr (kEnt) pr.w = __shfl_sync(0xFFFFFFFFu, o.w, r);
      acc = st_merge(acc, pr);
    }
    if (lane == 0) {
      row_state = acc;
      if (rank == 0) {
        if constexpr (kEnt)
          write_row_result(acc, xt, tvalid, T, c, logprob, lse, entropy, err, row);
        else
          write_row_result(acc, xt, tvalid, T, c, logprob, lse, err, row);
      }
    }
  }
  // no CTA may leave before the others have read its partial: arrive now
  // (relaxed: the reads above have returned their values), wait at the end
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
  __syncthreads();
  const St rs = row_state;
  if constexpr (kEnt) {
    // the entropy gradient from the lse and H just written (the same
    // expressions as write_row_result), as slp_bwd_kernel takes them
    float L20 = __int_as_float(0x7FC00000), Hl20 = L20;
    if (rs.m != -INFINITY && rs.s > 0.f) {
      const float l = rs.m / T + (log2f(rs.s) - fmaf(rs.m, c, -rs.mc)) * kLn2;
      const float H = (log2f(rs.s) - rs.w / rs.s) * kLn2;
      L20 = l * kLog2e;
      Hl20 = H * kLog2e;
    }
    BwdRow<Elt, true> b;
    b.set(tt, gT, L20, gH != nullptr ? dbg::ld(gH + row) * invT : 0.f, Hl20, c);
    const int64_t rel0 = static_cast<int64_t>(tt) - v0 * kVec;  // target offset in segment
    const int64_t tvec = rel0 >= 0 ? rel0 / kVec : -1;
    Elt* gr = gx + row * ldg;
    auto put = [&](int i, const uint4& v) {
      st_global_na(gv + i, b.vec(v));
      if (i == tvec) E::store1(gr + tt, b.one(E::load1(xr + tt), c, true));
    };
    for (int i = threadIdx.x; i < nv_s; i += kFbThreads) put(i, q[i]);
    if constexpr (kTV > 0) put_tmem<kTV>(taddr, nv_s, nv, put);
#pragma unroll
    for (int u = 0; u < kRV; ++u) {
      const int i = nv_r + u * kFbThreads + threadIdx.x;
      if (i < nv) put(i, rv[u]);
    }
    if (rank == C - 1)
      for (int64_t e = nvec * kVec + threadIdx.x; e < V; e += kFbThreads)
        E::store1(gr + e, b.one(E::load1(xr + e), c, e == tt));
    if constexpr (kTV > 0) free_tmem(tmem_holder);
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
    return;
  }

  // pass 2: gradient from shared memory.  p = 2^(x*c - off), off = mc + log2 s;
  // a p = sign(a) 2^(x*c - off + log2 |a|) (scaled_exp2_vec), the target's
  // element then rewritten by the thread that stored it.
  const float off = (rs.m == -INFINITY || !(rs.s > 0.f)) ? __int_as_float(0x7FC00000)
                                                          : rs.mc + log2f(rs.s);
  const float a = -gT;
  const float no1 = log2f(fabsf(a)) - off;
  const float2 cc = make_float2(c, c), no = make_float2(no1, no1);
  const uint32_t sgn = sign_mask(a, tag);
  const int64_t rel0 = static_cast<int64_t>(tt) - v0 * kVec;  // target offset in segment
  const int64_t tvec = rel0 >= 0 ? rel0 / kVec : -1;
  auto put = [&](int i, const uint4& v) {
    st_global_na(gv + i, scaled_exp2_vec(v, cc, no, sgn, tag));
    if (i == tvec) {
      const float p = ex2(fmaf(E::load1(xr + tt), c, -off));
      E::store1(gx + row * ldg + tt, fmaf(a, p, gT));
    }
  };
  for (int i = threadIdx.x; i < nv_s; i += kFbThreads) put(i, q[i]);
  if constexpr (kTV > 0) put_tmem<kTV>(taddr, nv_s, nv, put);
#pragma unroll
  for (int u = 0; u < kRV; ++u) {
    const int i = nv_r + u * kFbThreads + threadIdx.x;
    if (i < nv) put(i, rv[u]);
  }
  if (rank == C - 1) {
    for (int64_t e = nvec * kVec + threadIdx.x; e < V; e += kFbThreads) {
      const float p = ex2(fmaf(E::load1(xr + e), c, -off));
      E::store1(gx + row * ldg + e, (e == tt) ? fmaf(a, p, gT) : a * p);
    }
  }
  if constexpr (kTV > 0) free_tmem(tmem_holder);
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// ---- fused forward + backward, short rows: one warp per row ----------------
//
// A warp holds its row on chip: the first 32 * kNV vectors in registers (kNV
// per lane, plain 16-byte loads), the rest of a row longer than 8 KB in the
// warp's own slot of shared memory, filled by one bulk copy that lane 0
// issues before the register loads.  The lanes fold the log-sum-exp, merge by
// butterfly shuffles (every lane ends with the same state) and write the
// gradient from registers and shared memory.  No CTA barrier and no cluster:
// for short rows the per-row set-up of the cluster kernel above (barrier
// initialisation, CTA and cluster merges) costs more than the row's own
// traffic, and one CTA of 256 threads per 8 KB row keeps too few bytes in
// flight.
constexpr int kFbRowsWarps = 4;
constexpr int kFbRowsMaxNV = 16;                // register vectors per lane (8 KB per warp)
constexpr int kFbRowsMaxSlot = 24 * 1024;       // shared-memory part per warp
constexpr int kFbRowsMaxBytes = kFbRowsMaxNV * 32 * 16 + kFbRowsMaxSlot;  // 32 KB rows

// kEnt: with the entropy, as in slp_fwd_bwd_kernel (its 8-vector form needs
// more than 64 registers, so six CTAs per SM instead of eight).
template <typename Elt, int kNV, bool kEnt>
__global__ void __launch_bounds__(32 * kFbRowsWarps, kNV >= 16 ? 4 : (kEnt && kNV >= 8 ? 6 : 8))
    slp_fwd_bwd_rows_kernel(const Elt* __restrict__ x, int64_t N, int64_t V, int64_t ld,
                            const int32_t* __restrict__ t, const uint8_t* __restrict__ mask,
                            float T, float c, float invT, const float* __restrict__ g,
                            const float* __restrict__ gH, float* __restrict__ logprob,
                            float* __restrict__ lse, float* __restrict__ entropy,
                            Elt* __restrict__ gx, int64_t ldg, int32_t* __restrict__ err,
                            int slot_bytes SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  using E = Elem<Elt>;
  using St = typename std::conditional<kEnt, Lse3, Lse2>::type;
  constexpr int kVec = E::kVec;
  extern __shared__ __align__(128) uint8_t slots[];
  __shared__ __align__(8) uint64_t full[kFbRowsWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kFbRowsWarps + w;
  if (row >= N) return;
  const int64_t nvec = V / kVec;
  Elt* gr = gx + row * ldg;
  uint4* gv = reinterpret_cast<uint4*>(gr);
  if (mask != nullptr && dbg::ld(mask + row) == 0) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t i = lane; i < nvec; i += 32) st_stream(gv + i, z);
    for (int64_t e = nvec * kVec + lane; e < V; e += 32) E::store1(gr + e, 0.f);
    if (lane == 0) {
      dbg::st(logprob + row, 0.f);
      dbg::st(lse + row, 0.f);
      if (kEnt) dbg::st(entropy + row, 0.f);
    }
    return;
  }
  const Elt* xr = x + row * ld;
  const uint4* xv = reinterpret_cast<const uint4*>(xr);
  const int nreg = static_cast<int>(nvec < 32 * kNV ? nvec : 32 * kNV);
  const int ns = static_cast<int>(nvec - nreg);  // vectors in shared memory (<= slot_bytes / 16)
  const uint32_t slot = sm100::smem_u32(slots) + static_cast<uint32_t>(w * slot_bytes);
  const uint32_t bar = sm100::smem_u32(&full[w]);
  if (ns > 0) {
    if (lane == 0) {
      sm100::mbar_init(bar, 1);
      sm100::fence_mbar_init();
      sm100::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(ns) * 16u);
      sm100::bulk_load(slot, xv + nreg, static_cast<uint32_t>(ns) * 16u, bar);
    }
    __syncwarp();  // the barrier's initialisation is seen by every lane
  }
  const int32_t tt = dbg::ld(t + row);
  const bool tvalid = tt >= 0 && static_cast<int64_t>(tt) < V;
  const float gT = tvalid ? ((kEnt && g == nullptr) ? 0.f : dbg::ld(g + row) * invT)
                          : __int_as_float(0x7FC00000);
  const uint4 pad = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
  uint4 rv[kNV];
#pragma unroll
  for (int u = 0; u < kNV; ++u) {
    const int i = u * 32 + lane;
    rv[u] = i < nreg ? ld_stream(xv + i) : pad;
  }
  const Elt* tag = nullptr;
  St st;
  st_empty(st);
  if constexpr (kEnt)
    lse3_fold_vec<kNV>(st, rv, c, tag);
  else
    lse2_fold_vec<kNV>(st, rv, c, tag);
  const uint4* q = reinterpret_cast<const uint4*>(slots + w * slot_bytes);
  if (ns > 0) {
    bool ok = sm100::mbar_wait_bounded(bar, 0, nullptr, kFwdWaitNs);
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (!ok && lane == 0) {
      if (err != nullptr) atomicOr(err, SLP_DEVICE_ERR_TIMEOUT);
      sm100::mbar_wait_bounded(bar, 0, nullptr, kFwdWaitNs);  // let the copy land
    }
    constexpr int kPer = 4;
    for (int i0 = lane; i0 < ns; i0 += 32 * kPer) {
      uint4 vv[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = i0 + 32 * u;
        vv[u] = i < ns ? q[i] : pad;
      }
      if constexpr (kEnt)
        lse3_fold_vec<kPer>(st, vv, c, tag);
      else
        lse2_fold_vec<kPer>(st, vv, c, tag);
    }
  }
  for (int64_t e = nvec * kVec + lane; e < V; e += 32) {  // fewer than kVec trailing elements
    float f1[1] = {E::load1(xr + e)};
    st_fold<1>(st, f1, c);
  }
  st = st_warp_reduce(st);  // every lane holds the same state
  if (lane == 0) {
    const float xt = tvalid ? E::load1(xr + tt) : 0.f;
    if constexpr (kEnt)
      write_row_result(st, xt, tvalid, T, c, logprob, lse, entropy, err, row);
    else
      write_row_result(st, xt, tvalid, T, c, logprob, lse, err, row);
  }
  if constexpr (kEnt) {
    // the entropy gradient from the lse and H just written, as in
    // slp_fwd_bwd_kernel
    float L20 = __int_as_float(0x7FC00000), Hl20 = L20;
    if (st.m != -INFINITY && st.s > 0.f) {
      const float l = st.m / T + (log2f(st.s) - fmaf(st.m, c, -st.mc)) * kLn2;
      const float H = (log2f(st.s) - st.w / st.s) * kLn2;
      L20 = l * kLog2e;
      Hl20 = H * kLog2e;
    }
    BwdRow<Elt, true> b;
    b.set(tt, gT, L20, gH != nullptr ? dbg::ld(gH + row) * invT : 0.f, Hl20, c);
    const int64_t tvec = tvalid ? static_cast<int64_t>(tt) / kVec : -1;
    auto put = [&](int64_t i, const uint4& v) {
      st_stream(gv + i, b.vec(v));
      if (i == tvec) E::store1(gr + tt, b.one(E::load1(xr + tt), c, true));
    };
#pragma unroll
    for (int u = 0; u < kNV; ++u) {
      const int i = u * 32 + lane;
      if (i < nreg) put(i, rv[u]);
    }
    for (int i = lane; i < ns; i += 32) put(nreg + i, q[i]);
    for (int64_t e = nvec * kVec + lane; e < V; e += 32)
      E::store1(gr + e, b.one(E::load1(xr + e), c, e == tt));
    return;
  }

  // gradient, as in the cluster kernel: a p = sign(a) 2^(x c - off + log2 |a|)
  // per vector, the target's element rewritten by the lane that stored it
  const float off = (st.m == -INFINITY || !(st.s > 0.f)) ? __int_as_float(0x7FC00000)
                                                          : st.mc + log2f(st.s);
  const float a = -gT;
  const float no1 = log2f(fabsf(a)) - off;
  const float2 cc = make_float2(c, c), no = make_float2(no1, no1);
  const uint32_t sgn = sign_mask(a, tag);
  const int64_t tvec = tvalid ? static_cast<int64_t>(tt) / kVec : -1;
  auto put = [&](int64_t i, const uint4& v) {
    st_stream(gv + i, scaled_exp2_vec(v, cc, no, sgn, tag));
    if (i == tvec) {
      const float p = ex2(fmaf(E::load1(xr + tt), c, -off));
      E::store1(gr + tt, fmaf(a, p, gT));
    }
  };
#pragma unroll
  for (int u = 0; u < kNV; ++u) {
    const int i = u * 32 + lane;
    if (i < nreg) put(i, rv[u]);
  }
  for (int i = lane; i < ns; i += 32) put(nreg + i, q[i]);
  for (int64_t e = nvec * kVec + lane; e < V; e += 32) {
    const float p = ex2(fmaf(E::load1(xr + e), c, -off));
    E::store1(gr + e, (e == tt) ? fmaf(a, p, gT) : a * p);
  }
}

namespace {

bool aligned16(const void* p, int64_t ld, int esize) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ((ld * esize) & 15) == 0;
}

// CTAs per row of the ring forward (a cluster of that many CTAs when > 1).
// `ring` is the bytes one CTA keeps in flight; `per_sm` CTAs are resident per
// SM.  Measured (bf16, L2 flushed, one CTA per row against splits 2..8):
//  - When every row's CTA is resident at once, splitting only adds a
//    cluster's launch and barriers: N = 256, V = 151936: 26.2 us unsplit,
//    31.2 split 3, 34.0 split 4; V = 32768: 13.9 against 16.0.
//  - When the rows make a little more than one wave, a split evens out the
//    last wave for long rows: N = 512, V = 262144: 69.2 us split 2 against
//    75.3 unsplit; at V = 32768 a split leaves each CTA less than its ring
//    (18.4 unsplit against 23.0).
//  - From two waves on, one CTA per row ties or wins (N = 1024 and 2048 at
//    V = 32768, 151936, 262144).
// So: below one wave, the largest split that keeps every CTA resident; up to
// two waves, a split of 2; then none.  A CTA always gets at least one ring's
// worth of the row, and at most 8 CTAs (the portable cluster size) share it.
int choose_splits(int64_t N, int64_t row_bytes, int64_t ring, int per_sm) {
  const int64_t slots = static_cast<int64_t>(sm_count()) * per_sm;
  int64_t s = 1;
  if (N <= slots)
    s = slots / (N > 0 ? N : 1);
  else if (N < 2 * slots)
    s = 2;
  const int64_t by_len = row_bytes / ring;
  if (s > by_len) s = by_len;
  if (s > kMaxSplits) s = kMaxSplits;
  if (s < 1) s = 1;
  return static_cast<int>(s);
}

template <typename Elt, typename St>
cudaError_t fwd_typed(const Elt* x, int64_t N, int64_t V, int64_t ld, const int32_t* t,
                      const uint8_t* mask, float T, float* logprob, float* lse, float* entropy,
                      int32_t* err, cudaStream_t stream) {
  if (aligned16(x, ld, sizeof(Elt)) && use_rows_kernel(N, V * static_cast<int64_t>(sizeof(Elt)))) {
    const int64_t blocks = (N + kRowsWarps - 1) / kRowsWarps;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
    slp_fwd_rows_kernel<Elt, St><<<static_cast<unsigned>(blocks), 32 * kRowsWarps, 0, stream>>>(
        x, N, V, ld, t, mask, T, c, logprob, lse, entropy, err
        SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, sizeof(Elt)), {t, 4ull * N}, {mask, 1ull * N},
                            {logprob, 4ull * N}, {lse, 4ull * N}, {entropy, 4ull * N}}));
    return cudaGetLastError();
  }
  // 64 KB rings fit three CTAs per SM, 32 KB rings (with the entropy) six
  const int splits = choose_splits(N, V * static_cast<int64_t>(sizeof(Elt)), fwd_smem<St>(),
                                   fwd_stages<St>() == 4 ? 3 : 6);
  if (N * splits > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  const bool vec = aligned16(x, ld, sizeof(Elt));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(N * splits), 1, 1);
  cfg.blockDim = dim3(kFwdThreads, 1, 1);
  cfg.dynamicSmemBytes = vec ? fwd_smem<St>() : 0;
  cfg.stream = stream;
  if (vec) {
    cudaError_t e = cudaFuncSetAttribute(slp_fwd_kernel<Elt, true, St>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, fwd_smem<St>());
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[1];
  if (splits > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (vec)
    return cudaLaunchKernelEx(&cfg, slp_fwd_kernel<Elt, true, St>, x, V, ld, t, mask, T, c,
                              logprob, lse, entropy, err, splits
                              SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, sizeof(Elt)), {t, 4ull * N}, {mask, 1ull * N},
                            {logprob, 4ull * N}, {lse, 4ull * N}, {entropy, 4ull * N}}));
  return cudaLaunchKernelEx(&cfg, slp_fwd_kernel<Elt, false, St>, x, V, ld, t, mask, T, c, logprob,
                            lse, entropy, err, splits
                            SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, sizeof(Elt)), {t, 4ull * N}, {mask, 1ull * N},
                            {logprob, 4ull * N}, {lse, 4ull * N}, {entropy, 4ull * N}}));
}

// Rows of at most 64 KB that fill less than 90 % of their tiles of the
// backward's (row, tile) grid (16 KB tiles) take one warp per row.  Measured
// (bf16, N = 65536, TB/s, warp per row against the tile grid): 8 KB rows 6.78
// against 5.11, 12 KB 6.78 / 6.07, 20 KB 6.80 / 5.86, 40 KB 6.80 / 6.52; with
// full tiles the grid is ahead (16 KB 6.80 / 6.78 is a tie, 48 KB 6.67 / 6.87
// and 64 KB 6.60 / 6.92 at N = 16384).
constexpr bool use_bwd_rows_kernel(int64_t N, int64_t row_bytes) {
  constexpr int64_t kTileBytes = static_cast<int64_t>(kBwdThreads) * kBwdUnroll * 16;
  const int64_t tiles = (row_bytes + kTileBytes - 1) / kTileBytes;
  return N > 0 && row_bytes <= 64 * 1024 && row_bytes * 10 < tiles * kTileBytes * 9;
}

template <typename Elt, bool kEnt>
cudaError_t bwd_typed(const Elt* x, int64_t N, int64_t V, int64_t ld, const int32_t* t,
                      const uint8_t* mask, float T, const float* lse, const float* g,
                      const float* H, const float* gH, Elt* gx, int64_t ldg, int32_t* err,
                      cudaStream_t stream) {
  constexpr int64_t kTileElems =
      static_cast<int64_t>(kBwdThreads) * kBwdUnroll * Elem<Elt>::kVec;
  const int64_t tiles = (V + kTileElems - 1) / kTileElems;
  const int64_t blocks = N * tiles;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const float invT = 1.0f / T;
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  const bool vec = aligned16(x, ld, sizeof(Elt)) && aligned16(gx, ldg, sizeof(Elt));
  if (vec && use_bwd_rows_kernel(N, V * static_cast<int64_t>(sizeof(Elt)))) {
    const int64_t rblocks = (N + kRowsWarps - 1) / kRowsWarps;
    slp_bwd_rows_kernel<Elt, kEnt><<<static_cast<unsigned>(rblocks), 32 * kRowsWarps, 0, stream>>>(
        x, N, V, ld, t, mask, invT, c, lse, g, H, gH, gx, ldg, err
        SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, sizeof(Elt)), {t, 4ull * N}, {mask, 1ull * N},
                            {lse, 4ull * N}, {g, 4ull * N}, {H, 4ull * N}, {gH, 4ull * N},
                            dbg::rows(gx, N, V, ldg, sizeof(Elt))}));
    return cudaGetLastError();
  }
  if (vec)
    slp_bwd_kernel<Elt, true, kEnt><<<static_cast<unsigned>(blocks), kBwdThreads, 0, stream>>>(
        x, V, ld, t, mask, invT, c, lse, g, H, gH, gx, ldg, err, tiles
        SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, sizeof(Elt)), {t, 4ull * N}, {mask, 1ull * N},
                            {lse, 4ull * N}, {g, 4ull * N}, {H, 4ull * N}, {gH, 4ull * N},
                            dbg::rows(gx, N, V, ldg, sizeof(Elt))}));
  else
    slp_bwd_kernel<Elt, false, kEnt><<<static_cast<unsigned>(blocks), kBwdThreads, 0, stream>>>(
        x, V, ld, t, mask, invT, c, lse, g, H, gH, gx, ldg, err, tiles
        SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, sizeof(Elt)), {t, 4ull * N}, {mask, 1ull * N},
                            {lse, 4ull * N}, {g, 4ull * N}, {H, 4ull * N}, {gH, 4ull * N},
                            dbg::rows(gx, N, V, ldg, sizeof(Elt))}));
  return cudaGetLastError();
}

__host__ __device__ constexpr bool use_fb_rows_kernel(int64_t N, int64_t row_bytes) {
  return row_bytes <= kFbRowsMaxBytes && N > 0;
}

// gH and entropy are used with kEnt only.
template <typename Elt, int kNV, bool kEnt>
cudaError_t fwd_bwd_rows_launch(const Elt* x, int64_t N, int64_t V, int64_t ld, const int32_t* t,
                                const uint8_t* mask, float T, const float* g, const float* gH,
                                float* logprob, float* lse, float* entropy, Elt* gx, int64_t ldg,
                                int32_t* err, cudaStream_t stream) {
  constexpr int kVec = Elem<Elt>::kVec;
  const int64_t nvec = V / kVec;
  const int64_t ns = nvec > 32 * kNV ? nvec - 32 * kNV : 0;
  const int slot_bytes = static_cast<int>(ns * 16);
  if (slot_bytes > kFbRowsMaxSlot) return cudaErrorInvalidValue;
  const int smem = slot_bytes * kFbRowsWarps;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(slp_fwd_bwd_rows_kernel<Elt, kNV, kEnt>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kFbRowsMaxSlot * kFbRowsWarps);
    if (e != cudaSuccess) return e;
  }
  const int64_t blocks = (N + kFbRowsWarps - 1) / kFbRowsWarps;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  slp_fwd_bwd_rows_kernel<Elt, kNV, kEnt>
      <<<static_cast<unsigned>(blocks), 32 * kFbRowsWarps, smem, stream>>>(
          x, N, V, ld, t, mask, T, c, 1.0f / T, g, gH, logprob, lse, entropy, gx, ldg, err,
          slot_bytes SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, sizeof(Elt)), {t, 4ull * N}, {mask, 1ull * N},
                            {g, 4ull * N}, {gH, 4ull * N}, {logprob, 4ull * N}, {lse, 4ull * N},
                            {entropy, 4ull * N}, dbg::rows(gx, N, V, ldg, sizeof(Elt))}));
  return cudaGetLastError();
}

// Register vectors per lane: the smallest power of two that holds the row,
// at most kFbRowsMaxNV (the rest then goes to shared memory).
template <typename Elt, bool kEnt>
cudaError_t fwd_bwd_rows_typed(const Elt* x, int64_t N, int64_t V, int64_t ld, const int32_t* t,
                               const uint8_t* mask, float T, const float* g, const float* gH,
                               float* logprob, float* lse, float* entropy, Elt* gx, int64_t ldg,
                               int32_t* err, cudaStream_t stream) {
  const int64_t per_lane = (V / Elem<Elt>::kVec + 31) / 32;
#define SLP_FB_ROWS(NV)                                                                       \
  fwd_bwd_rows_launch<Elt, NV, kEnt>(x, N, V, ld, t, mask, T, g, gH, logprob, lse, entropy, gx, \
                                     ldg, err, stream)
  if (per_lane <= 1) return SLP_FB_ROWS(1);
  if (per_lane <= 2) return SLP_FB_ROWS(2);
  if (per_lane <= 4) return SLP_FB_ROWS(4);
  if (per_lane <= 8) return SLP_FB_ROWS(8);
  return SLP_FB_ROWS(16);
#undef SLP_FB_ROWS
}

// Whether the fused call runs the form with a TMEM part (C CTAs per row
// without it, C_tm with).  Rows longer than eight CTAs of the register form
// hold (about 606 KB) always take it: against the shared-memory-only clusters
// that served rows up to 768 KB, and the separate kernels beyond, it took 24
// to 29 % less time (703 KB rows: fp32 0.591 -> 0.450 ms, bf16 0.632 ->
// 0.475 ms; 1000 KB rows: 0.673 -> 0.480 and 0.689 -> 0.496 ms).  Shorter
// rows take it when they are fp32 and it saves at least two CTAs: fp32 rows
// of 65536 / 100000 / 131072 / 150000 columns (4 -> 2, 6 -> 3, 7 -> 4,
// 8 -> 5 CTAs) take 8 / 10 / 7 / 5 % less time, 75968 columns (4 -> 3) 1 %
// more.  On such bf16 rows, which carry twice the elements per byte, it lost
// (c151k 4 -> 3 CTAs: 0.414 against 0.396 ms; 248320 columns, 7 -> 4: 1.535
// against 1.443 ms): the TMEM part's loads, four vectors per round trip, and
// its fold come before the shared-memory chunks are consumed.
inline bool tmem_fused_form(int64_t C, int64_t C_tm, size_t esize) {
  if (C > kFbMaxCluster) return true;
  return esize == 4 && C_tm <= C - 2;
}

// Fused forward + backward: needs 16-byte-aligned rows and rows short enough
// to fit a cluster of at most 8 CTAs of the TMEM form (8 x kFbTmSeg bytes,
// about 1.1 MB); returns cudaErrorNotSupported
// otherwise (the caller then runs the separate kernels).  gH and entropy are
// used with kEnt only.
template <typename Elt, bool kEnt>
cudaError_t fwd_bwd_typed(const Elt* x, int64_t N, int64_t V, int64_t ld, const int32_t* t,
                          const uint8_t* mask, float T, const float* g, const float* gH,
                          float* logprob, float* lse, float* entropy, Elt* gx, int64_t ldg,
                          int32_t* err, cudaStream_t stream) {
  constexpr int kVec = Elem<Elt>::kVec;
  if (!aligned16(x, ld, sizeof(Elt)) || !aligned16(gx, ldg, sizeof(Elt)))
    return cudaErrorNotSupported;
  const int64_t nvec = V / kVec;
  if (use_fb_rows_kernel(N, V * static_cast<int64_t>(sizeof(Elt))))
    return fwd_bwd_rows_typed<Elt, kEnt>(x, N, V, ld, t, mask, T, g, gH, logprob, lse, entropy,
                                         gx, ldg, err, stream);
  // Segments of at most kFbRegSeg bytes (kFbRV vectors per thread in
  // registers, the rest in shared memory) keep four CTAs resident per SM;
  // with a TMEM part as well, a segment holds kFbTmSeg bytes, so long rows
  // need fewer CTAs per cluster.
  int64_t C = (nvec * 16 + kFbRegSeg - 1) / kFbRegSeg;
  if (C < 1) C = 1;
  const int64_t C_tm = (nvec * 16 + kFbTmSeg - 1) / kFbTmSeg;
  const bool tm = tmem_fused_form(C, C_tm, sizeof(Elt));
  if (tm) C = C_tm < 1 ? 1 : C_tm;
  if (C > kFbMaxCluster) return cudaErrorNotSupported;
  if (N * C > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const int64_t per = (nvec + C - 1) / C;  // vectors of the longest segment
  const int64_t on_chip = (kFbRV + (tm ? kFbTV : 0)) * kFbThreads;
  const int64_t in_smem = per > on_chip ? per - on_chip : 0;
  int smem = static_cast<int>(in_smem * 16);
  if (tm && smem < kFbTmMinSmem) smem = kFbTmMinSmem;
  auto kern = tm ? slp_fwd_bwd_kernel<Elt, kFbTV, kEnt> : slp_fwd_bwd_kernel<Elt, 0, kEnt>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kFbMaxSmem);
  if (e != cudaSuccess) return e;
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  const float invT = 1.0f / T;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(N * C), 1, 1);
  cfg.blockDim = dim3(kFbThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
  attr[1].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicyLoadBalancing;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, x, V, ld, t, mask, T, c, invT, g, gH, logprob, lse,
                            entropy, gx, ldg, err, static_cast<int>(C)
                            SLP_DBG_ARG(err, {dbg::rows(x, N, V, ld, sizeof(Elt)), {t, 4ull * N}, {mask, 1ull * N},
                            {g, 4ull * N}, {gH, 4ull * N}, {logprob, 4ull * N}, {lse, 4ull * N},
                            {entropy, 4ull * N}, dbg::rows(gx, N, V, ldg, sizeof(Elt))}));
}

}  // namespace

cudaError_t launch_forward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                           const int32_t* t, const uint8_t* mask, float T, float* logprob,
                           float* lse, int32_t* err, cudaStream_t stream) {
  if (dtype == SLP_BF16)
    return fwd_typed<__nv_bfloat16, Lse2>(static_cast<const __nv_bfloat16*>(x), N, V, ld, t, mask,
                                          T, logprob, lse, nullptr, err, stream);
  return fwd_typed<float, Lse2>(static_cast<const float*>(x), N, V, ld, t, mask, T, logprob, lse,
                                nullptr, err, stream);
}

cudaError_t launch_forward_entropy(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                   const int32_t* t, const uint8_t* mask, float T,
                                   float* logprob, float* lse, float* entropy, int32_t* err,
                                   cudaStream_t stream) {
  if (dtype == SLP_BF16)
    return fwd_typed<__nv_bfloat16, Lse3>(static_cast<const __nv_bfloat16*>(x), N, V, ld, t, mask,
                                          T, logprob, lse, entropy, err, stream);
  return fwd_typed<float, Lse3>(static_cast<const float*>(x), N, V, ld, t, mask, T, logprob, lse,
                                entropy, err, stream);
}

cudaError_t launch_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                            const int32_t* t, const uint8_t* mask, float T, const float* lse,
                            const float* grad_out, void* grad_x, int64_t ld_grad,
                            int32_t* err, cudaStream_t stream) {
  if (dtype == SLP_BF16)
    return bwd_typed<__nv_bfloat16, false>(static_cast<const __nv_bfloat16*>(x), N, V, ld, t,
                                           mask, T, lse, grad_out, nullptr, nullptr,
                                           static_cast<__nv_bfloat16*>(grad_x), ld_grad, err,
                                           stream);
  return bwd_typed<float, false>(static_cast<const float*>(x), N, V, ld, t, mask, T, lse,
                                 grad_out, nullptr, nullptr, static_cast<float*>(grad_x),
                                 ld_grad, err, stream);
}

cudaError_t launch_backward_entropy(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                    const int32_t* t, const uint8_t* mask, float T,
                                    const float* lse, const float* entropy,
                                    const float* grad_out, const float* grad_entropy,
                                    void* grad_x, int64_t ld_grad, int32_t* err,
                                    cudaStream_t stream) {
  // no entropy term: the plain backward, which then gives the same bits
  if (grad_entropy == nullptr && grad_out != nullptr)
    return launch_backward(x, dtype, N, V, ld, t, mask, T, lse, grad_out, grad_x, ld_grad, err,
                           stream);
  if (dtype == SLP_BF16)
    return bwd_typed<__nv_bfloat16, true>(static_cast<const __nv_bfloat16*>(x), N, V, ld, t,
                                          mask, T, lse, grad_out, entropy, grad_entropy,
                                          static_cast<__nv_bfloat16*>(grad_x), ld_grad, err,
                                          stream);
  return bwd_typed<float, true>(static_cast<const float*>(x), N, V, ld, t, mask, T, lse,
                                grad_out, entropy, grad_entropy, static_cast<float*>(grad_x),
                                ld_grad, err, stream);
}

cudaError_t launch_forward_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                    const int32_t* t, const uint8_t* mask, float T,
                                    const float* grad_out, float* logprob, float* lse,
                                    void* grad_x, int64_t ld_grad, int32_t* err,
                                    cudaStream_t stream) {
  cudaError_t e;
  if (dtype == SLP_BF16)
    e = fwd_bwd_typed<__nv_bfloat16, false>(static_cast<const __nv_bfloat16*>(x), N, V, ld, t,
                                            mask, T, grad_out, nullptr, logprob, lse, nullptr,
                                            static_cast<__nv_bfloat16*>(grad_x), ld_grad, err,
                                            stream);
  else
    e = fwd_bwd_typed<float, false>(static_cast<const float*>(x), N, V, ld, t, mask, T, grad_out,
                                    nullptr, logprob, lse, nullptr, static_cast<float*>(grad_x),
                                    ld_grad, err, stream);
  if (e != cudaErrorNotSupported) return e;
  // rows unaligned or too long for one cluster: the separate kernels
  e = launch_forward(x, dtype, N, V, ld, t, mask, T, logprob, lse, err, stream);
  if (e != cudaSuccess) return e;
  return launch_backward(x, dtype, N, V, ld, t, mask, T, lse, grad_out, grad_x, ld_grad, err,
                         stream);
}

cudaError_t launch_forward_backward_entropy(const void* x, int dtype, int64_t N, int64_t V,
                                            int64_t ld, const int32_t* t, const uint8_t* mask,
                                            float T, const float* grad_out,
                                            const float* grad_entropy, float* logprob, float* lse,
                                            float* entropy, void* grad_x, int64_t ld_grad,
                                            int32_t* err, cudaStream_t stream) {
  cudaError_t e;
  if (dtype == SLP_BF16)
    e = fwd_bwd_typed<__nv_bfloat16, true>(static_cast<const __nv_bfloat16*>(x), N, V, ld, t,
                                           mask, T, grad_out, grad_entropy, logprob, lse, entropy,
                                           static_cast<__nv_bfloat16*>(grad_x), ld_grad, err,
                                           stream);
  else
    e = fwd_bwd_typed<float, true>(static_cast<const float*>(x), N, V, ld, t, mask, T, grad_out,
                                   grad_entropy, logprob, lse, entropy,
                                   static_cast<float*>(grad_x), ld_grad, err, stream);
  if (e != cudaErrorNotSupported) return e;
  // rows unaligned or too long for one cluster: the separate kernels
  e = launch_forward_entropy(x, dtype, N, V, ld, t, mask, T, logprob, lse, entropy, err, stream);
  if (e != cudaSuccess) return e;
  return launch_backward_entropy(x, dtype, N, V, ld, t, mask, T, lse, entropy, grad_out,
                                 grad_entropy, grad_x, ld_grad, err, stream);
}

}  // namespace slp
