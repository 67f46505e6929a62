// Fused LM-head path: selected-token log-probabilities of z = h W^T / T
// without storing the logits, computing only rows whose loss mask is 1 (slime
// issue #2253, maintainer analysis: keep trainable rows before the vocabulary
// projection, compute compact rows, scatter scalars back).
//
// Forward
//   1. scan    : mask -> pos[N] (compact index or -1), idx[Na], Na     (1 CTA);
//                inactive rows get logprob = lse = 0
//   2. gather  : h_c[i] = h[idx[i]], rows Na..roundup(Na,256) zeroed
//   3. GEMM    : persistent tcgen05 kernel, 256 x 256 tiles of h_c W^T per
//                CTA pair with fp32 accumulators in TMEM; the epilogue warps
//                of each CTA keep an online
//                (max, sum-exp) per row over a slab of vocabulary tiles and
//                catch the target logit; one partial per (slab, row).  The
//                epilogue warp that stores the last slab of its 32 rows merges
//                their partials in slab order and writes logprob/lse to the
//                original rows.
// Backward, per vocabulary chunk of 16384 to V columns, as the caller's
// workspace allows (a bounded workspace instead of a [rows, V] buffer)
//   1-2. scan + gather as above (once)
//   3. GEMM (recompute): the chunk's tiles; the epilogue writes
//        dz = g/T (1[v == t] - 2^(x*c - lse*log2 e)) as bf16 (rows >= Na: 0)
//   4. GEMM dh_part[ks] = dz[:, K-slice] W[K-slice, :]  (split-K, fp32)
//   5. GEMM dW[chunk] = dz^T h_c (K = compact rows), bf16 stores; its idle
//        warps 2-3 meanwhile fold dh_acc (+)= sum_ks dh_part[ks] (fixed order)
//   then once: dh[r] = bf16(dh_acc[pos[r]]) (inactive rows 0)
//
// GEMM kernel layout: persistent, 256 threads per CTA, launched as clusters
// of two CTAs on two SMs (a CTA pair).  In each CTA warp 0 issues TMA loads
// of its 128 rows of A and its half of B into a 6-stage shared-memory ring
// (128-byte swizzle); warp 1 of the even CTA issues tcgen05.mma.cta_group::2
// (M=256 over both CTAs, N=256, K=16) into one of two TMEM accumulators --
// the whole warp runs the issue loop with warp-uniform operands and one
// elected lane issues, which keeps the issue well ahead of the tensor pipe
// (a one-lane branch issued about 80 cycles per MMA and starved it); warp 2
// owns the pair-wide TMEM allocation; warps 4-7 are the epilogue of their
// CTA's 128 rows (TMEM lane = row, so every row reduction is thread-local).
// Units (a row block's slab of vocabulary tiles, or one output tile) are
// handed out at run time: each pair claims the next one from a counter in
// the workspace and publishes it to every role of both CTAs through a small
// shared-memory ring.  Without pairs (a device that cannot co-schedule them, or
// SLP_LMHEAD_CTA_PAIRS=0) the same template runs one CTA per 128 x 256 tile
// with a 4-stage ring.  Every mbarrier wait gives up after its bound (two
// seconds by default), sets SLP_DEVICE_ERR_TIMEOUT, drains the copies and
// tensor-core work in flight and frees its TMEM instead of hanging.

#include "slp.h"
#include "slp_device.cuh"
#include "slp_internal.h"
#include "slp_sm100.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <stdlib.h>

#include <atomic>

namespace slp {
namespace lmh {

constexpr int BM = 128;   // rows of one CTA's tile (TMEM lanes)
constexpr int BN = 256;   // columns of a tile (TMEM columns per accumulator)
constexpr int BK = 64;    // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int A_BYTES = BM * BK * 2;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 2 * BN;
constexpr int kRowRound = 2 * BM;  // compact rows are padded to whole pair tiles

// Tile geometry of the two GEMM forms.  One CTA: a 128 x 256 tile per CTA.
// CTA pair (cta_group::2): a 256 x 256 tile per pair of CTAs on two SMs, one
// MMA instruction covering both; each CTA holds its 128 rows of A and half of
// B (128 tile columns), and its TMEM holds its 128 rows of the accumulator.
// For the same MMA work per SM a stage then carries 32 KB instead of 48 KB,
// which leaves room for more stages in flight.
template <bool kPair>
struct Tile {
  static constexpr int kCtas = kPair ? 2 : 1;
  static constexpr int kRows = BM * kCtas;        // rows of the (pair's) tile
  static constexpr int kBRows = BN / kCtas;       // B rows (tile columns) in one CTA
  static constexpr int kBBytes = kBRows * BK * 2;
  static constexpr int kStageBytes = A_BYTES + kBBytes;
  static constexpr int kStages = kPair ? 6 : 4;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 512 /*barriers*/;
};
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // default bound of a pipeline wait
constexpr uint64_t kDrainLimitNs = 2000000000ull;  // bound of the waits after a give-up
constexpr int kSlabCap = 256;  // most vocabulary slabs per row (forward partials)
constexpr int kWorkSlots = 8;  // units published ahead of the slowest consumer
constexpr int kKSplitCap = 24;  // most K splits of the dh GEMM
constexpr int kVChunk = 65536;     // vocabulary columns per backward chunk (default workspace)
constexpr int kVChunkMin = 16384;  // the narrowest chunk (smallest workspace)

enum Epi { EPI_LSE = 0, EPI_DZ = 1, EPI_F32 = 2, EPI_BF16 = 3, EPI_ACC32 = 4 };

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Work decomposition of one GEMM launch, a pure function of the sizes and of
// the grid, evaluated identically by every CTA and by the follow-up kernels.
struct Sched {
  int m_tiles, n_tiles, k_blocks, S, units;
  int bm;  // rows of one tile (128 for one CTA, 256 for a CTA pair)
};

// Slabs of vocabulary tiles per row block: the S minimising the tile count of
// the busiest CTA (ties -> fewer slabs, i.e. fewer partials).
__host__ __device__ inline int choose_slabs(int m_tiles, int n_tiles, int G) {
  int best = 1;
  long long best_cost = -1;
  const int smax = n_tiles < kSlabCap ? n_tiles : kSlabCap;
  for (int S = 1; S <= smax; ++S) {
    const long long cost = static_cast<long long>(cdiv(m_tiles * S, G)) * cdiv(n_tiles, S);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

// K splits of the dh GEMM: the fewest splits (at least s_min, so that one
// K-slice of W stays in L2 while every row block reads it) whose busiest CTA
// is within 3 % of the best balance.  Fewer splits mean less partial storage
// and less partial traffic for the accumulation.
__host__ __device__ inline int choose_ksplits(int tiles, int k_blocks, int G, int s_min) {
  int lo = s_min < 1 ? 1 : s_min;
  if (lo > kKSplitCap) lo = kKSplitCap;
  if (lo > k_blocks) lo = k_blocks > 0 ? k_blocks : 1;
  const int hi = k_blocks < kKSplitCap ? (k_blocks > 0 ? k_blocks : 1) : kKSplitCap;
  long long best_cost = -1;
  for (int S = lo; S <= hi; ++S) {
    const long long cost = static_cast<long long>(cdiv(tiles * S, G)) * cdiv(k_blocks, S);
    if (best_cost < 0 || cost < best_cost) best_cost = cost;
  }
  for (int S = lo; S <= hi; ++S) {
    const long long cost = static_cast<long long>(cdiv(tiles * S, G)) * cdiv(k_blocks, S);
    if (cost * 100 <= best_cost * 103) return S;
  }
  return lo;
}

__host__ __device__ inline int ksplit_min(int V, int d) {
  // keep a K-slice of W under ~48 MB (a third of L2)
  const long long bytes = static_cast<long long>(V) * d * 2;
  return static_cast<int>((bytes + (48ll << 20) - 1) / (48ll << 20));
}

// bm: rows of one tile.  G: tiles in flight at once (CTAs, or CTA pairs).
// f32_cap: floats of split-K partial storage available to the dh GEMM; the
// split count is clamped to it (fewer splits are still a correct schedule).
__host__ __device__ inline Sched make_sched(int epi, int Na, int V, int d, int G, int bm,
                                            long long f32_cap = -1) {
  Sched s{};
  s.bm = bm;
  if (epi == EPI_LSE || epi == EPI_DZ) {
    s.m_tiles = cdiv(Na, bm);
    s.n_tiles = cdiv(V, BN);
    s.k_blocks = d / BK;
    s.S = choose_slabs(s.m_tiles, s.n_tiles, G);
    s.units = s.m_tiles * s.S;
  } else if (epi == EPI_F32) {
    s.m_tiles = cdiv(Na, bm);
    s.n_tiles = cdiv(d, BN);
    s.k_blocks = cdiv(V, BK);
    s.S = choose_ksplits(s.m_tiles * s.n_tiles, s.k_blocks, G, ksplit_min(V, d));
    if (f32_cap >= 0 && s.m_tiles > 0) {
      const long long per_split = static_cast<long long>(s.m_tiles) * bm * d;
      const long long smax = f32_cap / per_split;
      if (s.S > smax) s.S = smax < 1 ? 1 : static_cast<int>(smax);
    }
    s.units = s.m_tiles * s.n_tiles * s.S;
  } else {
    s.m_tiles = cdiv(V, bm);
    s.n_tiles = cdiv(d, BN);
    s.k_blocks = cdiv(Na, BM) * (BM / BK);  // compact rows Na..roundup(Na, 128) are zero
    s.S = 1;
    s.units = s.m_tiles * s.n_tiles;
  }
  return s;
}

struct Unit {
  int m, n0, n1, k0, k1, slab;
};

__device__ __forceinline__ Unit decode(const Sched& s, int epi, int u) {
  Unit w;
  if (epi == EPI_LSE || epi == EPI_DZ) {
    w.slab = u / s.m_tiles;
    w.m = u - w.slab * s.m_tiles;
    w.n0 = static_cast<int>(static_cast<long long>(w.slab) * s.n_tiles / s.S);
    w.n1 = static_cast<int>(static_cast<long long>(w.slab + 1) * s.n_tiles / s.S);
    w.k0 = 0;
    w.k1 = s.k_blocks;
  } else if (epi == EPI_F32) {
    const int mn = s.m_tiles * s.n_tiles;
    w.slab = u / mn;  // K split
    const int r = u - w.slab * mn;
    w.m = r / s.n_tiles;
    w.n0 = r - w.m * s.n_tiles;
    w.n1 = w.n0 + 1;
    w.k0 = static_cast<int>(static_cast<long long>(w.slab) * s.k_blocks / s.S);
    w.k1 = static_cast<int>(static_cast<long long>(w.slab + 1) * s.k_blocks / s.S);
  } else {
    w.slab = 0;
    w.m = u / s.n_tiles;
    w.n0 = u - w.m * s.n_tiles;
    w.n1 = w.n0 + 1;
    w.k0 = 0;
    w.k1 = s.k_blocks;
  }
  return w;
}

struct Params {
  int V;                      // vocabulary columns of this launch (a backward chunk)
  int d, N, Mcap;
  int v0;                     // first vocabulary column of this launch
  int Vtot;                   // whole vocabulary (valid targets are [0, Vtot))
  int G;                      // grid size the schedule was made for
  const int32_t* counters;    // [0] = Na; [1], [2]: unit counters of alternate launches
  const int32_t* idx;         // compact row -> original row
  const int32_t* t;           // [N] targets
  const float* g;             // [N] upstream gradient (backward)
  const float* lse;           // [N] saved lse (backward)
  float c;                    // log2(e) / T
  float invT;
  float4* part;               // [kSlabCap][Mcap] forward partials {m, mc, s, x_t}
  __nv_bfloat16* dz;          // [Mcap][ld_dz]
  long long ld_dz;
  float* part_f32;            // [S][Mpad][d] split-K partials of dh (Mpad from Na)
  float* dh_acc;              // [Mcap][d] fp32 dh accumulated over the chunks
  int dh_fold;                // dW launches: warps 2-3 fold this chunk's dh partials into dh_acc
  long long pf32_cap;         // floats available at part_f32
  __nv_bfloat16* out;         // dW [V][d] (this launch's rows)
  float* out_acc;             // fp32 dW accumulated into (EPI_ACC32)
  int32_t* err;
  int32_t* row_cnt;           // [Mcap / BM][4] slab counters of the forward GEMM (zeroed by the scan)
  float* out_lp;              // forward results [N] (original rows)
  float* out_lse;
  float T;
  unsigned long long wait_ns;  // bound of every pipeline wait (after it: give up, flag, drain)
  int32_t* work;               // units claimed so far beyond the first G (zero at launch)
  int32_t* work_next;          // the next launch's counter, zeroed by this one
};

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float (&v)[32]) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = v[q * 8 + j];
    dbg::st(d4 + q, Elem<__nv_bfloat16>::pack(f));
  }
}

// v[i] for a run-time i in [0, 32) as a tree of selects on the bits of i, so
// the 32 values stay in registers (no indexed local-memory copy).
__device__ __forceinline__ float select32(const float (&v)[32], int i) {
  float a[16], b[8], c[4], d[2];
#pragma unroll
  for (int j = 0; j < 16; ++j) a[j] = (i & 16) ? v[j + 16] : v[j];
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = (i & 8) ? a[j + 8] : a[j];
#pragma unroll
  for (int j = 0; j < 4; ++j) c[j] = (i & 4) ? b[j + 4] : b[j];
#pragma unroll
  for (int j = 0; j < 2; ++j) d[j] = (i & 2) ? c[j + 2] : c[j];
  return (i & 1) ? d[1] : d[0];
}

template <int kEpi, bool kAmn, bool kBmn, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    lmh_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const Params p SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  using namespace sm100;
  using TL = Tile<kPair>;
  constexpr int STAGES = TL::kStages;
  constexpr int STAGE_BYTES = TL::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5 + 2 * kWorkSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* peer_fills = reinterpret_cast<volatile int*>(tmem_holder + 2);
  volatile int* work_ring = reinterpret_cast<volatile int*>(tmem_holder + 4);  // [kWorkSlots]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar_full = smem_u32(bars);
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_accf = bar_full + 16 * STAGES;
  const uint32_t bar_acce = bar_accf + 16;
  const uint32_t bar_done = bar_acce + 16;  // the MMA thread's last commit
  const uint32_t bar_wfull = bar_done + 8;  // [kWorkSlots] a unit published in the slot
  const uint32_t bar_wempty = bar_wfull + 8 * kWorkSlots;  // [kWorkSlots] slot read by all
  const uint32_t ring = smem_u32(smem);
  // The pair: rank 0 issues the MMAs and owns the barriers the MMA thread
  // waits on (full, accumulator-empty); both CTAs load, and both drain their
  // own TMEM rows.  Without a pair the same code runs with rank 0 alone.
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int tile0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tiles_in_flight = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const uint32_t lead_full = kPair ? mapa_rank(bar_full, 0) : bar_full;
  const uint32_t lead_acce = kPair ? mapa_rank(bar_acce, 0) : bar_acce;
  const uint32_t peer_abort =
      kPair ? mapa_rank(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u) : 0u;
  const uint32_t lead_wempty = kPair ? mapa_rank(bar_wempty, 0) : bar_wempty;
  // a wait that gave up here ends the other CTA's waits too
  auto give_up = [&]() {
    *abort_flag = 1;
    if (kPair) st_cluster_u32(peer_abort, 1u);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_accf + 8 * b, 1);
      mbar_init(bar_acce + 8 * b, 4 * TL::kCtas);  // one arrival per epilogue warp of the pair
    }
    mbar_init(bar_done, 1);
    // Unit hand-out: rank 0's producer publishes each unit into the ring of
    // both CTAs; every consumer of the pair (the other producer, the MMA
    // thread, the epilogue warps) frees the slot on rank 0 once it has read it.
    for (int j = 0; j < kWorkSlots; ++j) {
      mbar_init(bar_wfull + 8 * j, 1);
      mbar_init(bar_wempty + 8 * j, 1 + 4 * TL::kCtas + (kPair ? 1 : 0));
    }
    *abort_flag = 0;
    *peer_fills = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 2) {
    if (kPair)
      tmem_alloc_pair(smem_u32(tmem_holder), kTmemCols);
    else
      tmem_alloc(smem_u32(tmem_holder), kTmemCols);
  }
  tc_fence_before();
  if (kPair) {
    __syncwarp();
    pair_sync();  // both CTAs' barriers exist before either signals the other's
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int Na = dbg::ld(p.counters);
  const Sched sc = make_sched(kEpi, Na, p.V, p.d, p.G, TL::kRows, p.pf32_cap);
  int fills = 0;  // stage fills this CTA's producer issued
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.work_next != nullptr) dbg::st(p.work_next, 0);

  // Units: each pair starts with unit tile0 (its index), so every pair has
  // one however few units there are, then claims the next unclaimed unit from
  // a global counter, one ahead of the unit it works on (so the atomic's
  // latency hides behind the unit in progress); pairs that run faster take
  // more units.  (Claiming the first unit as well let the first pairs to
  // start take two units each when there were about as many units as pairs,
  // and the last ones none.)  Every role of both CTAs walks the same
  // sequence: work item wi sits in slot wi % kWorkSlots; -1 ends it.  (Waits
  // on it acquire at cluster scope: the publishing arrival may come from the
  // other CTA.)
  auto take_unit = [&](int wi, int& u) -> bool {
    if (!mbar_wait_bounded<kPair>(bar_wfull + 8 * (wi % kWorkSlots), (wi / kWorkSlots) & 1,
                                  abort_flag, p.wait_ns))
      return false;
    u = work_ring[wi % kWorkSlots];
    return true;
  };
  auto free_slot = [&](int wi) {
    if (kPair)
      mbar_arrive_cluster(lead_wempty + 8 * (wi % kWorkSlots));
    else
      mbar_arrive(bar_wempty + 8 * (wi % kWorkSlots));
  };
  auto claim_unit = [&]() -> int {
    return dbg::ok(p.work, 4) ? atomicAdd(p.work, 1) + tiles_in_flight : sc.units;
  };

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      int u = tile0;  // rank 0: the unit to publish next; rank 1: overwritten by the ring
      int claim = sc.units;
      if (rank == 0 && u < sc.units) claim = claim_unit();
      for (int wi = 0; ok; ++wi) {
        const int slot = wi % kWorkSlots;
        if (rank == 0) {
          // publish unit u (or the end) once every consumer has read the slot's last one
          if (!mbar_wait_bounded<kPair>(bar_wempty + 8 * slot, ((wi / kWorkSlots) & 1) ^ 1,
                                        abort_flag, p.wait_ns)) {
            give_up();
            break;
          }
          const int item = u < sc.units ? u : -1;
          work_ring[slot] = item;
          if (kPair) {
            st_cluster_u32(mapa_rank(smem_u32(const_cast<int*>(work_ring + slot)), 1),
                           static_cast<uint32_t>(item));
            mbar_arrive_cluster(mapa_rank(bar_wfull + 8 * slot, 1));
          }
          mbar_arrive(bar_wfull + 8 * slot);
          u = item;
        } else {
          if (!take_unit(wi, u)) {
            give_up();
            break;
          }
          free_slot(wi);
        }
        if (u < 0) break;
        const Unit w = decode(sc, kEpi, u);
        const int arow = w.m * TL::kRows + static_cast<int>(rank) * BM;  // this CTA's A rows
        for (int n = w.n0; n < w.n1 && ok; ++n) {
          const int bcol = n * BN + static_cast<int>(rank) * TL::kBRows;  // this CTA's B rows
          for (int kb = w.k0; kb < w.k1; ++kb, ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            if (!mbar_wait_bounded(bar_empty + 8 * s, ph ^ 1, abort_flag, p.wait_ns)) {
              give_up();
              ok = false;
              break;
            }
            // rank 0 expects the bytes of both CTAs on its own full barrier
            if (rank == 0) mbar_arrive_expect_tx(bar_full + 8 * s, STAGE_BYTES * TL::kCtas);
            const uint32_t fb = lead_full + 8 * s;
            const uint32_t a_dst = ring + s * STAGE_BYTES;
            const uint32_t b_dst = a_dst + A_BYTES;
            auto load = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1) {
              if (kPair)
                tma_load_2d_pair(dst, m, c0, c1, fb);
              else
                tma_load_2d(dst, m, c0, c1, fb);
            };
            if (!kAmn) {
              load(a_dst, &tmA, kb * BK, arow);
            } else {
#pragma unroll
              for (int j = 0; j < BM / 64; ++j) load(a_dst + j * 8192, &tmA, arow + 64 * j, kb * BK);
            }
            if (!kBmn) {
              load(b_dst, &tmB, kb * BK, bcol);
            } else {
#pragma unroll
              for (int j = 0; j < TL::kBRows / 64; ++j)
                load(b_dst + j * 8192, &tmB, bcol + 64 * j, kb * BK);
            }
          }
        }
        if (rank == 0) {
          u = claim;
          if (u < sc.units) claim = claim_unit();
        }
      }
      fills = it;
      if (!kPair) {
        // Drain: wait (bounded, ignoring the abort flag) for the copies issued
        // into the last STAGES slots, so no copy lands in shared memory after
        // the CTA has exited.  Earlier copies were consumed: their slots were
        // refilled only after the MMAs reading them finished.  After a normal
        // run these phases have completed already (the MMA thread waited on
        // them); after a give-up anywhere in the CTA some may still be landing.
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          mbar_wait_bounded(bar_full + 8 * (j % STAGES), (j / STAGES) & 1, nullptr,
                            kDrainLimitNs);
      } else if (rank == 1) {
        // tell rank 0, which drains the pair's copies after the cluster barrier
        st_cluster_u32(mapa_rank(smem_u32(const_cast<int*>(peer_fills)), 0), static_cast<uint32_t>(it));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (rank 0 only) ----------------
    // The whole warp runs this loop; every wait is agreed by the warp, and
    // one elected lane issues each MMA and commit (inside the helpers).
    if (rank == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(TL::kRows, BN, kAmn, kBmn);
      int it = 0, tc = 0;
      bool ok = true;
      for (int wi = 0; ok; ++wi) {
        int u = -1;
        if (!__all_sync(0xFFFFFFFFu, take_unit(wi, u))) {
          if (lane == 0) give_up();
          break;
        }
        u = __shfl_sync(0xFFFFFFFFu, u, 0);
        if (lane == 0) free_slot(wi);
        if (u < 0) break;
        const Unit w = decode(sc, kEpi, u);
        for (int n = w.n0; n < w.n1 && ok; ++n, ++tc) {
          const int buf = tc & 1;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_acce + 8 * buf,
                                                         ((tc >> 1) & 1) ^ 1, abort_flag,
                                                         p.wait_ns))) {
            if (lane == 0) give_up();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          for (int kb = w.k0; kb < w.k1; ++kb, ++it) {
            const int s = it % STAGES;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_full + 8 * s, (it / STAGES) & 1,
                                                           abort_flag, p.wait_ns))) {
              if (lane == 0) give_up();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = ring + s * STAGE_BYTES;
            const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t ad = kAmn ? umma_desc_sw128(a_addr + k * 2048, 8192, 1024)
                                       : umma_desc_sw128(a_addr + k * 32, 16, 1024);
              const uint64_t bd = kBmn ? umma_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                       : umma_desc_sw128(b_addr + k * 32, 16, 1024);
              if (kPair)
                mma_bf16_pair(d_tmem, ad, bd, idesc, (kb > w.k0 || k > 0) ? 1u : 0u);
              else
                mma_bf16(d_tmem, ad, bd, idesc, (kb > w.k0 || k > 0) ? 1u : 0u);
            }
            // frees the stage (in both CTAs) once these MMAs finish
            if (kPair)
              mma_commit_pair_mc(bar_empty + 8 * s, 3);
            else
              mma_commit(bar_empty + 8 * s);
          }
          if (!ok) break;
          // accumulator ready for the epilogue (of both CTAs)
          if (kPair)
            mma_commit_pair_mc(bar_accf + 8 * buf, 3);
          else
            mma_commit(bar_accf + 8 * buf);
        }
      }
      // Every MMA the warp issued has completed before the CTA barrier
      // below, so none still writes TMEM when warp 2 frees it.  After a
      // normal run the epilogue has waited for all of them already; after a
      // give-up (here or in the epilogue) some may still be running.
      if (it > 0) {
        if (kPair)
          mma_commit_pair(bar_done);
        else
          mma_commit(bar_done);
        mbar_wait_bounded(bar_done, 0, nullptr, kDrainLimitNs);
      }
    }
  } else if ((kEpi == EPI_BF16 || kEpi == EPI_ACC32) && warp < 4) {
    // ------- warps 2-3 of a dW launch: dh split-K fold (tensor pipe idle) -------
    // dh_acc[i] (first chunk: =, later: +=) sum over the K splits of the dh
    // GEMM that ran just before, in split order, for every compact row i < Na.
    // The dW GEMM does not touch dh_acc or the partials, so the two overlap.
    if (p.dh_fold) {
      const Sched sf = make_sched(EPI_F32, Na, p.V, p.d, p.G, TL::kRows, p.pf32_cap);
      const long long mpad = static_cast<long long>(sf.m_tiles) * sf.bm;
      const bool first = p.v0 == 0;
      const int nw = static_cast<int>(gridDim.x) * 2;
      for (int i = static_cast<int>(blockIdx.x) * 2 + (warp - 2); i < Na; i += nw) {
        float* acc = p.dh_acc + static_cast<long long>(i) * p.d;
        for (int j0 = lane * 4; j0 < p.d; j0 += 512) {
          float4 a[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j0 + 128 * k < p.d && !first)
              a[k] = dbg::ld(reinterpret_cast<const float4*>(acc + j0 + 128 * k));
          }
          for (int sp = 0; sp < sf.S; ++sp) {
            const float* src = p.part_f32 + (sp * mpad + i) * p.d + j0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if (j0 + 128 * k >= p.d) continue;
              const float4 v = dbg::ld(reinterpret_cast<const float4*>(src + 128 * k));
              a[k].x += v.x;
              a[k].y += v.y;
              a[k].z += v.z;
              a[k].w += v.w;
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (j0 + 128 * k < p.d) dbg::st(reinterpret_cast<float4*>(acc + j0 + 128 * k), a[k]);
        }
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs: each drains its own TMEM rows) ----------------
    const int q = warp & 3;
    const int rit = q * 32 + lane;  // row within this CTA's 128 rows = TMEM lane
    int tc = 0;
    bool ok = true;
    for (int wi = 0; ok; ++wi) {
      // every lane waits and reads; the warp frees the slot once
      int u = -1;
      const bool got = take_unit(wi, u);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        if (lane == 0) give_up();
        break;
      }
      __syncwarp();
      if (lane == 0) free_slot(wi);
      if (u < 0) break;
      const Unit w = decode(sc, kEpi, u);
      const int rblk = w.m * TL::kCtas + static_cast<int>(rank);  // 128-row block of this CTA
      const int row = rblk * BM + rit;
      // per-row constants
      bool valid = false;
      int tr = -1;
      float coef = 0.f, L2 = 0.f;
      Lse2 st = lse2_empty();
      float xt = __int_as_float(0x7FC00000);
      if (kEpi == EPI_LSE || kEpi == EPI_DZ) {
        valid = row < Na;
        if (valid) {
          const int orig = dbg::ld(p.idx + row);
          tr = dbg::ld(p.t + orig);
          if (tr < 0 || tr >= p.Vtot) {
            tr = -1;  // invalid target: no gradient contribution, flagged elsewhere
            valid = kEpi == EPI_LSE;
          } else {
            tr -= p.v0;  // column within this launch (may fall outside it)
            if (kEpi == EPI_DZ) {
              coef = dbg::ld(p.g + orig) * p.invT;
              L2 = dbg::ld(p.lse + orig) * kLog2e;
            }
          }
        }
      }
      for (int n = w.n0; n < w.n1; ++n, ++tc) {
        const int buf = tc & 1;
        // every lane waits; the warp then agrees, so no lane reaches the
        // warp-wide tcgen05.ld alone
        const bool got = mbar_wait_bounded(bar_accf + 8 * buf, (tc >> 1) & 1, abort_flag,
                                           p.wait_ns);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          if (lane == 0) give_up();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
        const bool empty_k = w.k1 <= w.k0;
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
          uint32_t r[32];
          tmem_ld_32cols(taddr + ch * 32, r);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = empty_k ? 0.f : __uint_as_float(r[j]);
          const int col0 = n * BN + ch * 32;
          if (kEpi == EPI_LSE) {
            if (col0 + 32 > p.V) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j >= p.V) v[j] = -INFINITY;
            }
            if (tr >= col0 && tr < col0 + 32) xt = select32(v, tr - col0);
            if (col0 < p.V) lse2_fold<32>(st, v, p.c);
          } else if (kEpi == EPI_DZ) {
            if (col0 < p.V) {
              float o[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float pr = ex2(fmaf(v[j], p.c, -L2));
                o[j] = (col0 + j == tr) ? fmaf(-coef, pr, coef) : -coef * pr;
                if (!valid) o[j] = 0.f;
              }
              __nv_bfloat16* dst = p.dz + static_cast<long long>(row) * p.ld_dz + col0;
              if (col0 + 32 <= p.V) {
                store_bf16x32(dst, o);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (col0 + j < p.V) dbg::st(dst + j, __float2bfloat16_rn(o[j]));
              }
            }
          } else if (kEpi == EPI_F32) {
            if (row < Na && col0 < p.d) {
              const long long mpad = static_cast<long long>(sc.m_tiles) * sc.bm;
              float* dst = p.part_f32 + (static_cast<long long>(w.slab) * mpad + row) * p.d + col0;
              float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                dbg::st(d4 + j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
            }
          } else if (kEpi == EPI_BF16) {
            if (row < p.V && col0 < p.d)
              store_bf16x32(p.out + static_cast<long long>(row) * p.d + col0, v);
          } else {  // EPI_ACC32: dW += this micro-batch's gradient, in fp32
            if (row < p.V && col0 < p.d) {
              float4* d4 = reinterpret_cast<float4*>(p.out_acc + static_cast<long long>(row) * p.d + col0);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                float4 o = dbg::ld(d4 + j);
                o.x += v[4 * j];
                o.y += v[4 * j + 1];
                o.z += v[4 * j + 2];
                o.w += v[4 * j + 3];
                dbg::st(d4 + j, o);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (kPair)
            mbar_arrive_cluster(lead_acce + 8 * buf);
          else
            mbar_arrive(bar_acce + 8 * buf);
        }
      }
      if (kEpi == EPI_LSE && ok) {
        if (valid)
          dbg::st(p.part + static_cast<long long>(w.slab) * p.Mcap + row,
                  make_float4(st.m, st.mc, st.s, xt));
        // Each epilogue warp counts its 32 rows' slabs; the warp completing
        // the count (the last slab to store them) merges the S partials of
        // each row in slab order and writes the row's results.
        __threadfence();
        __syncwarp();
        int* cnt = p.row_cnt + rblk * 4 + q;
        int old = 0;
        if (lane == 0 && dbg::ok(cnt, 4)) old = atomicAdd(cnt, 1);
        old = __shfl_sync(0xFFFFFFFFu, old, 0);
        if (old == sc.S - 1 && row < Na) {
          __threadfence();
          const int orig = dbg::ld(p.idx + row);
          const int tt = dbg::ld(p.t + orig);
          const bool tvalid = tt >= 0 && tt < p.Vtot;
          const int ttile = tvalid ? tt / BN : -1;
          Lse2 acc = lse2_empty();
          float xtr = 0.f;
          // eight slabs' partials in flight at a time, merged in slab order
          constexpr int kBatch = 8;
          for (int s0 = 0; s0 < sc.S; s0 += kBatch) {
            float4 pv[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
              pv[j] = s0 + j < sc.S
                          ? dbg::ldcg(p.part + static_cast<long long>(s0 + j) * p.Mcap + row)
                          : make_float4(-INFINITY, -INFINITY, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
              const int sl = s0 + j;
              if (sl >= sc.S) break;
              acc = lse2_merge(acc, Lse2{pv[j].x, pv[j].y, pv[j].z});
              const int n0 = static_cast<int>(static_cast<long long>(sl) * sc.n_tiles / sc.S);
              const int n1 = static_cast<int>(static_cast<long long>(sl + 1) * sc.n_tiles / sc.S);
              if (ttile >= n0 && ttile < n1) xtr = pv[j].w;
            }
          }
          write_row_result(acc, xtr, tvalid, p.T, p.c, p.out_lp, p.out_lse, p.err, orig);
        }
      }
    }
  }

  tc_fence_before();
  if (kPair) {
    // Both CTAs are done issuing.  Rank 0 then drains every copy of the pair
    // still landing: each CTA's copies count on rank 0's full barriers, and
    // neither CTA may exit while a copy into either's shared memory, or onto
    // rank 0's barriers, is in flight.
    __syncwarp();
    pair_sync();
    if (rank == 0 && warp == 0 && lane == 0) {
      const int mine = fills;
      const int peer = *peer_fills;
      const int hi = mine > peer ? mine : peer;
      for (int j = (hi > STAGES ? hi - STAGES : 0); j < hi; ++j) {
        const uint32_t fb = bar_full + 8 * (j % STAGES);
        if (j >= mine)
          mbar_arrive_expect_tx(fb, STAGE_BYTES);  // the peer's half only: rank 0 never armed it
        else if (j >= peer)
          mbar_complete_tx(fb, STAGE_BYTES);  // armed for both halves; the peer's never comes
        mbar_wait_bounded(fb, (j / STAGES) & 1, nullptr, kDrainLimitNs);
      }
    }
    __syncwarp();
    pair_sync();
  } else {
    __syncthreads();
  }
  if (warp == 2) {
    tc_fence_after();
    if (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag && p.err != nullptr) atomicOr(p.err, SLP_DEVICE_ERR_TIMEOUT);
}

// ---- compaction ---------------------------------------------------------------

__global__ void __launch_bounds__(1024)
    lmh_scan_kernel(const uint8_t* __restrict__ mask, int N, int32_t* __restrict__ counters,
                    int32_t* __restrict__ pos, int32_t* __restrict__ idx,
                    int32_t* __restrict__ row_cnt, int n_row_cnt, float* __restrict__ lp0,
                    float* __restrict__ lse0 SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  // One CTA; each thread takes kRows consecutive rows per pass, so a pass
  // covers 8192 rows with one block-wide scan of the per-thread counts.
  constexpr int kRows = 8;
  __shared__ int warp_sums[32];
  __shared__ int carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int j = threadIdx.x; j < n_row_cnt; j += blockDim.x) dbg::st(row_cnt + j, 0);
  if (threadIdx.x == 0) {
    carry = 0;
    dbg::st(counters + 1, 0);  // unit counters of the GEMM launches that follow
    dbg::st(counters + 2, 0);
  }
  __syncthreads();
  for (int base = 0; base < N; base += 1024 * kRows) {
    const int r0 = base + threadIdx.x * kRows;
    int f[kRows];
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < kRows; ++e) {
      const int r = r0 + e;
      f[e] = (r < N) && (mask == nullptr || dbg::ld(mask + r) != 0) ? 1 : 0;
      cnt += f[e];
    }
    int v = cnt;  // inclusive scan of the counts across the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    int excl = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + v - cnt;
#pragma unroll
    for (int e = 0; e < kRows; ++e) {
      const int r = r0 + e;
      if (r >= N) break;
      if (f[e]) {
        dbg::st(pos + r, excl);
        dbg::st(idx + excl, r);
        ++excl;
      } else {
        dbg::st(pos + r, -1);
        if (lp0 != nullptr) {  // forward: inactive rows give zeros
          dbg::st(lp0 + r, 0.f);
          dbg::st(lse0 + r, 0.f);
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_sums[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) dbg::st(counters, static_cast<int32_t>(carry));
}

// Warp w of the grid copies active row w of h to its compact slot; warps
// N .. N+255 zero compact rows Na .. roundup(Na, 256)-1 (whole pair tiles).
constexpr int kGatherWarps = 8;
__global__ void __launch_bounds__(32 * kGatherWarps)
    lmh_gather_kernel(const __nv_bfloat16* __restrict__ h, int N, int d,
                      const int32_t* __restrict__ counters, const int32_t* __restrict__ pos,
                      __nv_bfloat16* __restrict__ hc SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  const int w = static_cast<int>(blockIdx.x) * kGatherWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int nv = d / 8;  // 16-byte vectors per row
  int dst_row;
  const uint4* src = nullptr;
  if (w < N) {
    dst_row = dbg::ld(pos + w);
    if (dst_row < 0) return;
    src = reinterpret_cast<const uint4*>(h + static_cast<long long>(w) * d);
  } else if (w < N + kRowRound) {
    const int Na = dbg::ld(counters);
    dst_row = Na + (w - N);
    if (dst_row >= cdiv(Na, kRowRound) * kRowRound) return;
  } else {
    return;
  }
  uint4* dst = reinterpret_cast<uint4*>(hc + static_cast<long long>(dst_row) * d);
  for (int i0 = lane; i0 < nv; i0 += 32 * 4) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + 32 * u;
      v[u] = (src != nullptr && i < nv) ? dbg::ld(src + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + 32 * u < nv) dbg::st(dst + i0 + 32 * u, v[u]);
  }
}

// ---- dh: the final scatter ---------------------------------------------------------

// dh[r] = bf16(dh_acc[pos[r]]); inactive rows 0; rows with a bad target NaN.
__global__ void __launch_bounds__(256)
    lmh_dh_finish_kernel(const Params p, const int32_t* __restrict__ pos,
                         __nv_bfloat16* __restrict__ dh SLP_DBG_PARAM) {
  SLP_DBG_ENTER();
  const int r = blockIdx.x;
  const int i = dbg::ld(pos + r);
  __nv_bfloat16* out = dh + static_cast<long long>(r) * p.d;
  const int tt = dbg::ld(p.t + r);
  const bool bad = i >= 0 && (tt < 0 || tt >= p.Vtot);
  if (bad && threadIdx.x == 0 && p.err != nullptr) atomicOr(p.err, SLP_DATA_ERR_TARGET);
  for (int j = threadIdx.x * 4; j < p.d; j += blockDim.x * 4) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i >= 0) a = dbg::ld(reinterpret_cast<const float4*>(p.dh_acc + static_cast<long long>(i) * p.d + j));
    if (bad) a.x = a.y = a.z = a.w = __int_as_float(0x7FC00000);
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&lo);
    w.y = *reinterpret_cast<uint32_t*>(&hi);
    dbg::st(reinterpret_cast<uint2*>(out + j), w);
  }
}

// ---- host side ------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  // looked up once (thread-safe static initialisation); NULL if unavailable
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return nullptr;
  }();
  return fn;
}

// 2-D bf16 tensor [outer][inner] (row stride row_bytes), 128-byte swizzled box
// of box_inner x box_outer elements; reads outside the tensor return zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
              uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

template <int kEpi, bool kAmn, bool kBmn, bool kPair>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const Params& p,
                        cudaStream_t stream SLP_DBG_PARAM) {
  using TL = Tile<kPair>;
  auto k = lmh_gemm_kernel<kEpi, kAmn, kBmn, kPair>;
  cudaError_t e =
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, TL::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (!kPair) {
    k<<<p.G, kThreads, TL::kSmemBytes, stream>>>(a, b, p SLP_DBG_PASS(slp_dbg_bounds));
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * p.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = TL::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a, b, p SLP_DBG_PASS(slp_dbg_bounds));
}

// How the GEMMs run on the current device: as CTA pairs (cta_group::2),
// one pair per two SMs that the device can co-schedule as a cluster, or as
// one CTA per SM when it cannot.  G = tiles in flight (pairs or CTAs), bm =
// rows of one tile.  Queried once per device; the workspace layout and every
// launch use the same answer.
struct Geometry {
  bool pair;
  int G;
  int bm;
};

Geometry geometry() {
  // per device, filled on first use: pairs that fit, or -1 for none (or not
  // wanted); threads that race here store the same value
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int pairs = cached[dev].load(std::memory_order_relaxed);
  if (pairs == 0) {
    // SLP_LMHEAD_CTA_PAIRS=0 in the environment keeps the one-CTA form (read
    // once per device, at the first LM-head call or workspace query)
    const char* env = getenv("SLP_LMHEAD_CTA_PAIRS");
    int n = 0;
    if (env == nullptr || env[0] != '0') {
      auto k = lmh_gemm_kernel<EPI_LSE, false, false, true>;
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Tile<true>::kSmemBytes) == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2 * (sm_count() / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = Tile<true>::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) n = 0;
      }
      cudaGetLastError();  // a failed query leaves no sticky error behind
    }
    pairs = n > 0 ? n : -1;
    cached[dev].store(pairs, std::memory_order_relaxed);
  }
  if (pairs > 0) return Geometry{true, pairs, Tile<true>::kRows};
  return Geometry{false, sm_count(), Tile<false>::kRows};
}

struct Layout {
  Geometry geo;
  int Mcap;
  int vchunk;          // vocabulary columns per backward chunk
  long long ld_dz;     // row stride of the dz chunk buffer
  size_t off_counters, off_rcnt, off_pos, off_idx, off_hc, off_part, fwd_end;
  size_t off_dz, off_pf32, off_acc, bwd_end;
};

// Largest split-K partial footprint S * roundup(Na, bm) * d over every
// Na <= N and both chunk widths, for the geometry the kernels will use.
size_t max_partial_floats(int Mcap, int V, int vchunk, int d, const Geometry& g) {
  size_t best = 0;
  const int widths[2] = {vchunk < V ? vchunk : V, V % vchunk == 0 ? (vchunk < V ? vchunk : V)
                                                                 : V % vchunk};
  for (int w = 0; w < 2; ++w)
    for (int mt = 1; mt * g.bm <= Mcap; ++mt) {
      const Sched sc = make_sched(EPI_F32, mt * g.bm, widths[w], d, g.G, g.bm);
      const size_t f = static_cast<size_t>(sc.S) * mt * g.bm * d;
      if (f > best) best = f;
    }
  return best;
}

// vchunk: the backward's vocabulary chunk width (the whole vocabulary when
// V is smaller).
Layout layout(int64_t N, int64_t V, int64_t d, int64_t vchunk = kVChunk) {
  Layout L{};
  L.geo = geometry();
  L.Mcap = static_cast<int>(cdiv(static_cast<int>(N), kRowRound) * kRowRound);
  L.vchunk = V < vchunk ? static_cast<int>(V) : static_cast<int>(vchunk);
  L.ld_dz = (L.vchunk + 63) / 64 * 64;
  size_t o = 0;
  L.off_counters = o; o += 256;
  L.off_rcnt = o; o = align256(o + 4 * static_cast<size_t>(L.Mcap / BM) * 4);
  L.off_pos = o; o = align256(o + 4 * static_cast<size_t>(N));
  L.off_idx = o; o = align256(o + 4 * static_cast<size_t>(L.Mcap));
  L.off_hc = o; o = align256(o + 2 * static_cast<size_t>(L.Mcap) * d);
  L.off_part = o; o = align256(o + 16 * static_cast<size_t>(kSlabCap) * L.Mcap);
  L.fwd_end = o;
  L.off_dz = L.off_part;  // the backward does not use the forward partials
  o = align256(L.off_dz + 2 * static_cast<size_t>(L.Mcap) * L.ld_dz);
  L.off_pf32 = o;
  size_t pf = max_partial_floats(L.Mcap, static_cast<int>(V), L.vchunk, static_cast<int>(d), L.geo);
  if (vchunk == kVChunkMin) {
    // the smallest workspace also caps the split-K partials at two splits of
    // every row; the dh GEMM then takes fewer splits (a correct schedule with
    // less balance) wherever its best one would need more
    const size_t cap = 2 * static_cast<size_t>(L.Mcap) * d;
    if (pf > cap) pf = cap;
  }
  o = align256(o + 4 * pf);
  L.off_acc = o; o = align256(o + 4 * static_cast<size_t>(L.Mcap) * d);
  L.bwd_end = o > L.fwd_end ? o : L.fwd_end;
  return L;
}

// One GEMM launch in the layout's geometry.
template <int kEpi, bool kAmn, bool kBmn>
cudaError_t launch(const Layout& L, const CUtensorMap& a, const CUtensorMap& b, const Params& p,
                   cudaStream_t stream SLP_DBG_PARAM) {
  return L.geo.pair ? launch_gemm<kEpi, kAmn, kBmn, true>(a, b, p, stream
                                                         SLP_DBG_PASS(slp_dbg_bounds))
                    : launch_gemm<kEpi, kAmn, kBmn, false>(a, b, p, stream
                                                          SLP_DBG_PASS(slp_dbg_bounds));
}

// Bound of the pipeline waits for the launches that follow (process-wide).
std::atomic<unsigned long long> g_wait_ns{kWaitLimitNs};

// The j-th GEMM launch of a call counts its units on counters[1 + j % 2] and
// zeroes the other for launch j + 1 (the scan zeroes both first).
inline void set_launch(Params& p, int j) {
  int32_t* c = const_cast<int32_t*>(p.counters);
  p.work = c + 1 + (j & 1);
  p.work_next = c + 1 + ((j + 1) & 1);
}

struct Prepared {
  Layout L;
  Params p;
  int32_t* pos;
  __nv_bfloat16* hc;
  SLP_DBG_ONLY(dbg::Bounds bnd;)  // the call's buffers and the workspace sections it uses
};

#ifdef SLP_DEBUG_BOUNDS
void dbg_add(dbg::Bounds& b, const void* p, size_t bytes) {
  if (p != nullptr && bytes > 0 && b.n < dbg::kMaxRanges) b.r[b.n++] = dbg::Range{p, bytes};
}
#endif

// The widest backward chunk whose workspace fits in ws_bytes: the whole
// vocabulary, then 131072, 65536 (the default), 32768 or 16384 columns.  A
// narrower chunk needs a smaller dz chunk and fewer split-K partials, for
// more launch boundaries.
int64_t chunk_for(int64_t N, int64_t V, int64_t d, size_t ws_bytes) {
  const int64_t widths[4] = {V, 2ll * kVChunk, kVChunk, kVChunk / 2};
  for (int64_t w : widths)
    if (layout(N, V, d, w).bwd_end <= ws_bytes) return w;
  return kVChunkMin;
}

// logprob / lse: the forward's outputs (their inactive rows are zeroed here),
// NULL for the backward.
cudaError_t prepare(const void* h, int64_t N, int64_t V, int64_t d, const int32_t* t,
                    const uint8_t* mask, float T, void* ws, int32_t* err, cudaStream_t stream,
                    Prepared* out, float* logprob = nullptr, float* lse = nullptr,
                    int64_t vchunk = kVChunk) {
  Prepared& P = *out;
  P.L = layout(N, V, d, vchunk);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* counters = reinterpret_cast<int32_t*>(w + P.L.off_counters);
  P.pos = reinterpret_cast<int32_t*>(w + P.L.off_pos);
  int32_t* idx = reinterpret_cast<int32_t*>(w + P.L.off_idx);
  P.hc = reinterpret_cast<__nv_bfloat16*>(w + P.L.off_hc);
  Params& p = P.p;
  p = Params{};
  p.V = static_cast<int>(V);
  p.Vtot = static_cast<int>(V);
  p.v0 = 0;
  p.d = static_cast<int>(d);
  p.N = static_cast<int>(N);
  p.Mcap = P.L.Mcap;
  p.G = P.L.geo.G;
  p.counters = counters;
  p.idx = idx;
  p.t = t;
  p.c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  p.invT = 1.0f / T;
  p.part = reinterpret_cast<float4*>(w + P.L.off_part);
  p.dz = reinterpret_cast<__nv_bfloat16*>(w + P.L.off_dz);
  p.ld_dz = P.L.ld_dz;
  p.part_f32 = reinterpret_cast<float*>(w + P.L.off_pf32);
  p.dh_acc = reinterpret_cast<float*>(w + P.L.off_acc);
  p.pf32_cap = static_cast<long long>((P.L.off_acc - P.L.off_pf32) / 4);
  p.err = err;
  p.row_cnt = reinterpret_cast<int32_t*>(w + P.L.off_rcnt);
  p.out_lp = logprob;
  p.out_lse = lse;
  p.T = T;
  p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  set_launch(p, 0);
#ifdef SLP_DEBUG_BOUNDS
  {
    const uint64_t n = static_cast<uint64_t>(N);
    P.bnd = dbg::make(err, {{h, 2 * n * d}, {t, 4 * n}, {mask, n}, {logprob, 4 * n},
                            {lse, 4 * n}});
    const Layout& L = P.L;
    auto sec = [&](size_t lo, size_t hi) { dbg_add(P.bnd, w + lo, hi - lo); };
    sec(L.off_counters, L.off_rcnt);
    sec(L.off_rcnt, L.off_pos);
    sec(L.off_pos, L.off_idx);
    sec(L.off_idx, L.off_hc);
    sec(L.off_hc, L.off_part);
    if (logprob != nullptr) {  // forward: the slab partials
      sec(L.off_part, L.fwd_end);
    } else {  // backward: dz chunk, split-K partials, dh accumulator
      sec(L.off_dz, L.off_pf32);
      sec(L.off_pf32, L.off_acc);
      sec(L.off_acc, L.bwd_end);
    }
  }
#endif
  lmh_scan_kernel<<<1, 1024, 0, stream>>>(mask, p.N, counters, P.pos, idx, p.row_cnt,
                                          (P.L.Mcap / BM) * 4, logprob, lse
                                          SLP_DBG_PASS(P.bnd));
  lmh_gather_kernel<<<cdiv(p.N + kRowRound, kGatherWarps), 32 * kGatherWarps, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(h), p.N, p.d, counters, P.pos, P.hc
      SLP_DBG_PASS(P.bnd));
  return cudaGetLastError();
}

}  // namespace lmh

uint64_t lmhead_set_wait_limit(uint64_t ns) {
  return lmh::g_wait_ns.exchange(ns == 0 ? lmh::kWaitLimitNs : ns);
}

size_t lmhead_forward_workspace_size(int64_t N, int64_t V, int64_t d) {
  return lmh::layout(N, V, d).fwd_end;
}

size_t lmhead_workspace_size(int64_t N, int64_t V, int64_t d) {
  return lmh::layout(N, V, d).bwd_end;
}

size_t lmhead_workspace_size_max(int64_t N, int64_t V, int64_t d) {
  return lmh::layout(N, V, d, V).bwd_end;
}

size_t lmhead_workspace_size_min(int64_t N, int64_t V, int64_t d) {
  return lmh::layout(N, V, d, lmh::kVChunkMin).bwd_end;
}

cudaError_t launch_lmhead_forward(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                                  const int32_t* t, const uint8_t* mask, float T, float* logprob,
                                  float* lse, void* ws, int32_t* err, cudaStream_t stream) {
  using namespace lmh;
  Prepared P;
  cudaError_t e = prepare(h, N, V, d, t, mask, T, ws, err, stream, &P, logprob, lse);
  if (e != cudaSuccess) return e;
  const uint32_t brows = static_cast<uint32_t>(BN / (P.L.geo.pair ? 2 : 1));  // B rows per CTA
  CUtensorMap ma, mb;
  if (!make_map(&ma, P.hc, d, P.L.Mcap, d * 2, BK, BM) ||
      !make_map(&mb, W, d, V, d * 2, BK, brows))
    return cudaErrorInvalidValue;
  SLP_DBG_ONLY(dbg_add(P.bnd, W, 2ull * V * d);)
  return launch<EPI_LSE, false, false>(P.L, ma, mb, P.p, stream SLP_DBG_PASS(P.bnd));
}

cudaError_t launch_lmhead_backward(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                                   const int32_t* t, const uint8_t* mask, float T,
                                   const float* lse, const float* grad_out, void* dh, void* dW,
                                   void* ws, size_t ws_bytes, int32_t* err, cudaStream_t stream,
                                   bool accumulate_f32) {
  using namespace lmh;
  Prepared P;
  cudaError_t e = prepare(h, N, V, d, t, mask, T, ws, err, stream, &P, nullptr, nullptr,
                          chunk_for(N, V, d, ws_bytes));
  if (e != cudaSuccess) return e;
  P.p.g = grad_out;
  P.p.lse = lse;
#ifdef SLP_DEBUG_BOUNDS
  dbg_add(P.bnd, W, 2ull * V * d);
  dbg_add(P.bnd, grad_out, 4ull * N);
  dbg_add(P.bnd, lse, 4ull * N);
  dbg_add(P.bnd, dh, 2ull * N * d);
  dbg_add(P.bnd, dW, (accumulate_f32 ? 4ull : 2ull) * V * d);
#endif
  CUtensorMap m_hc_k, m_hc_mn;
  if (!make_map(&m_hc_k, P.hc, d, P.L.Mcap, d * 2, BK, BM) ||    // A of recompute
      !make_map(&m_hc_mn, P.hc, d, P.L.Mcap, d * 2, 64, BK))     // B of dW (N = d)
    return cudaErrorInvalidValue;
  const uint64_t dz_row = static_cast<uint64_t>(P.L.ld_dz) * 2;
  const __nv_bfloat16* Wb = static_cast<const __nv_bfloat16*>(W);
  int j = 0;  // GEMM launches so far
  for (int64_t v0 = 0; v0 < V; v0 += P.L.vchunk) {
    const int64_t vc = V - v0 < P.L.vchunk ? V - v0 : P.L.vchunk;
    Params pc = P.p;
    pc.v0 = static_cast<int>(v0);
    pc.V = static_cast<int>(vc);
    if (accumulate_f32)
      pc.out_acc = static_cast<float*>(dW) + v0 * d;
    else
      pc.out = static_cast<__nv_bfloat16*>(dW) + v0 * d;
    const __nv_bfloat16* Wc = Wb + v0 * d;
    CUtensorMap m_w_k, m_dz_k, m_w_mn, m_dz_mn;
    const uint32_t brows = static_cast<uint32_t>(BN / (P.L.geo.pair ? 2 : 1));
    if (!make_map(&m_w_k, Wc, d, vc, d * 2, BK, brows) ||             // B of recompute
        !make_map(&m_dz_k, pc.dz, vc, P.L.Mcap, dz_row, BK, BM) ||    // A of dh (K = chunk)
        !make_map(&m_w_mn, Wc, d, vc, d * 2, 64, BK) ||               // B of dh (N = d)
        !make_map(&m_dz_mn, pc.dz, vc, P.L.Mcap, dz_row, 64, BK))     // A of dW (M = chunk)
      return cudaErrorInvalidValue;
    set_launch(pc, j++);
    e = launch<EPI_DZ, false, false>(P.L, m_hc_k, m_w_k, pc, stream SLP_DBG_PASS(P.bnd));
    if (e != cudaSuccess) return e;
    set_launch(pc, j++);
    e = launch<EPI_F32, false, true>(P.L, m_dz_k, m_w_mn, pc, stream SLP_DBG_PASS(P.bnd));
    if (e != cudaSuccess) return e;
    set_launch(pc, j++);
    pc.dh_fold = 1;
    e = accumulate_f32
            ? launch<EPI_ACC32, true, true>(P.L, m_dz_mn, m_hc_mn, pc, stream SLP_DBG_PASS(P.bnd))
            : launch<EPI_BF16, true, true>(P.L, m_dz_mn, m_hc_mn, pc, stream SLP_DBG_PASS(P.bnd));
    if (e != cudaSuccess) return e;
  }
  lmh_dh_finish_kernel<<<static_cast<int>(N), 256, 0, stream>>>(
      P.p, P.pos, static_cast<__nv_bfloat16*>(dh) SLP_DBG_PASS(P.bnd));
  return cudaGetLastError();
}

}  // namespace slp
