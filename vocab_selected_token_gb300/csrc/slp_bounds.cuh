// Bounds-checked build of libslp, standing in for a memory checker.
//
// Built with -DSLP_DEBUG_BOUNDS, every kernel takes one more parameter: the
// byte ranges of the buffers its call was given (the inputs, outputs and
// workspace sections, each sized from the call's N, V, d and row strides).
// At entry thread 0 copies them into a per-CTA shared-memory table, and every
// global load and store of the kernel is checked against that table before it
// is made: an access must lie wholly inside one range.  An access outside all
// of them is skipped (a load returns zero bits), and SLP_DEVICE_ERR_BOUNDS is
// ORed into the call's error word.  Nothing traps.  A bulk copy is checked on
// its source range; a refused copy completes its mbarrier transaction by hand
// so the pipeline does not stall.  TMA tiled loads are bounded by their
// tensor maps, whose extents are set from the call's sizes, so they need no
// check.  Without the flag all of this compiles to nothing: the parameter,
// the table and the checks disappear.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "slp.h"

#ifdef SLP_DEBUG_BOUNDS
#include <initializer_list>
#endif

namespace slp {
namespace dbg {

constexpr int kMaxRanges = 20;

struct Range {
  const void* p;
  unsigned long long bytes;
};

struct Bounds {
  Range r[kMaxRanges];
  int n;
  int32_t* err;
};

#ifdef SLP_DEBUG_BOUNDS

// Host: the table of one launch.  Null pointers and empty ranges are left
// out; ranges beyond kMaxRanges are dropped (and would then fail closed: the
// accesses to them are reported).
inline Bounds make(int32_t* err, std::initializer_list<Range> rs) {
  Bounds b{};
  b.err = err;
  for (const Range& r : rs)
    if (r.p != nullptr && r.bytes > 0 && b.n < kMaxRanges) b.r[b.n++] = r;
  if (err != nullptr && b.n < kMaxRanges) b.r[b.n++] = Range{err, 4};
  return b;
}

// Byte range of `rows` rows of `cols` elements at row stride `ld` elements.
inline Range rows(const void* p, long long rows_, long long cols, long long ld, int esize) {
  if (p == nullptr || rows_ <= 0 || cols <= 0) return Range{nullptr, 0};
  return Range{p, static_cast<unsigned long long>(((rows_ - 1) * ld + cols) * esize)};
}

static __shared__ Bounds g_table;

__device__ __forceinline__ void enter(const Bounds& b) {
  if (threadIdx.x == 0) g_table = b;
  __syncthreads();
}

__device__ __forceinline__ bool ok(const void* p, unsigned long long bytes) {
  const unsigned long long a = reinterpret_cast<unsigned long long>(p);
  for (int i = 0; i < g_table.n; ++i) {
    const unsigned long long lo = reinterpret_cast<unsigned long long>(g_table.r[i].p);
    if (a >= lo && a + bytes <= lo + g_table.r[i].bytes) return true;
  }
  if (g_table.err != nullptr) atomicOr(g_table.err, SLP_DEVICE_ERR_BOUNDS);
  return false;
}

#define SLP_DBG_PARAM , const ::slp::dbg::Bounds slp_dbg_bounds
#define SLP_DBG_ENTER() ::slp::dbg::enter(slp_dbg_bounds)
#define SLP_DBG_ARG(...) , ::slp::dbg::make(__VA_ARGS__)
#define SLP_DBG_PASS(b) , (b)
#define SLP_DBG_ONLY(...) __VA_ARGS__

#else

__device__ __forceinline__ constexpr bool ok(const void*, unsigned long long) { return true; }

#define SLP_DBG_PARAM
#define SLP_DBG_ENTER() ((void)0)
#define SLP_DBG_ARG(...)
#define SLP_DBG_PASS(b)
#define SLP_DBG_ONLY(...)

#endif

// Checked plain accesses: in the checked build a refused load gives T{} and a
// refused store is skipped; otherwise they are the plain accesses.
template <typename T>
__device__ __forceinline__ T ld(const T* p) {
  return ok(p, sizeof(T)) ? *p : T{};
}

template <typename T>
__device__ __forceinline__ void st(T* p, const T& v) {
  if (ok(p, sizeof(T))) *p = v;
}

template <typename T>
__device__ __forceinline__ T ldcg(const T* p) {
  return ok(p, sizeof(T)) ? __ldcg(p) : T{};
}

}  // namespace dbg
}  // namespace slp
