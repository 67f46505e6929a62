// Host-resident logits: slp_forward_backward streamed through the GPU in row
// chunks.  Host code only (copies, events, launches of the fused kernel).
//
// Per device the library keeps two copy streams (host -> device, device ->
// host) and a ring of kHostSlots chunk buffers in the caller's workspace.
// Chunk k's inputs are copied on the in-stream, computed on the caller's
// stream, and its results copied back on the out-stream; events order each
// slot's reuse, so the three stages of consecutive chunks overlap.

#include "slp.h"
#include "slp_internal.h"

#include <cuda_runtime.h>
#include <mutex>
#include <vector>
#include <stdint.h>

namespace slp {
namespace {

constexpr int kHostSlots = 3;
constexpr int kMaxDevices = 64;
constexpr int64_t kDefaultChunkBytes = 64ll << 20;

struct CopyStreams {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t entry = nullptr, done = nullptr;
  cudaEvent_t in_done[kHostSlots] = {}, cmp_done[kHostSlots] = {}, out_done[kHostSlots] = {};
};

std::mutex g_mu;  // one enqueue at a time: the events below are shared per device
CopyStreams g_cs[kMaxDevices];

cudaError_t copy_streams(CopyStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CopyStreams& c = g_cs[dev];
  if (!c.ready) {
    e = cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.entry, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.done, cudaEventDisableTiming);
    for (int s = 0; s < kHostSlots && e == cudaSuccess; ++s) {
      e = cudaEventCreateWithFlags(&c.in_done[s], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.cmp_done[s], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.out_done[s], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return e;
    c.ready = true;
  }
  *out = &c;
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace: the per-row vectors of all N rows (copied in once, and out once
// at the end, so each chunk moves only its two big blocks), then the ring of
// slots, each holding one chunk's logits and gradient.
struct HostLayout {
  size_t t, g, m, lp, lse, slots;  // offsets
  size_t slot_bytes, slot_gx;      // slot size, gradient offset within a slot
};

HostLayout host_layout(int64_t N, int64_t V, int esize, int64_t R) {
  HostLayout L{};
  const size_t n = static_cast<size_t>(N > 0 ? N : 0);
  size_t o = 0;
  L.t = o; o = align256(o + n * 4);
  L.g = o; o = align256(o + n * 4);
  L.m = o; o = align256(o + n);
  L.lp = o; o = align256(o + n * 4);
  L.lse = o; o = align256(o + n * 4);
  L.slots = o;
  const size_t block = align256(static_cast<size_t>(R) * V * esize);
  L.slot_gx = block;
  L.slot_bytes = 2 * block;
  return L;
}

// Chunk plan: equal chunks of rows_per_chunk rows (0: about 64 MB of logits
// per chunk, which measured best against 16, 32 and 128 MB, and against a
// plan that ramped from 8 MB chunks up to 64 MB and down again).  Returns the
// largest chunk (the slot size in rows).
int64_t chunk_plan(int64_t N, int64_t V, int esize, int64_t rows_per_chunk,
                   std::vector<int64_t>* sizes) {
  int64_t R = rows_per_chunk > 0 ? rows_per_chunk : kDefaultChunkBytes / (V * esize);
  if (R < 1) R = 1;
  if (R > N && N > 0) R = N;
  sizes->clear();
  for (int64_t r0 = 0; r0 < N; r0 += R) sizes->push_back(N - r0 < R ? N - r0 : R);
  if (sizes->empty()) sizes->push_back(0);
  return R;
}

}  // namespace

size_t forward_backward_host_workspace_size(int64_t N, int64_t V, int esize,
                                            int64_t rows_per_chunk) {
  std::vector<int64_t> plan;
  const int64_t R = chunk_plan(N, V, esize, rows_per_chunk, &plan);
  HostLayout L = host_layout(N, V, esize, R);
  const int slots = plan.size() < kHostSlots ? static_cast<int>(plan.size()) : kHostSlots;
  return L.slots + slots * L.slot_bytes;
}

cudaError_t launch_forward_backward_host(const void* x_host, int dtype, int64_t N, int64_t V,
                                         int64_t ld, const int32_t* t_host,
                                         const uint8_t* mask_host, float T, const float* g_host,
                                         float* lp_host, float* lse_host, void* gx_host,
                                         int64_t ld_grad, int64_t rows_per_chunk, void* ws,
                                         int32_t* err, cudaStream_t stream) {
  const int esize = dtype == SLP_BF16 ? 2 : 4;
  std::vector<int64_t> plan;
  const int64_t R = chunk_plan(N, V, esize, rows_per_chunk, &plan);
  const int64_t chunks = static_cast<int64_t>(plan.size());
  const HostLayout L = host_layout(N, V, esize, R);
  const size_t row_bytes = static_cast<size_t>(V) * esize;
  char* w = static_cast<char*>(ws);
  int32_t* td = reinterpret_cast<int32_t*>(w + L.t);
  float* gd = reinterpret_cast<float*>(w + L.g);
  uint8_t* md = mask_host != nullptr ? reinterpret_cast<uint8_t*>(w + L.m) : nullptr;
  float* lpd = reinterpret_cast<float*>(w + L.lp);
  float* lsed = reinterpret_cast<float*>(w + L.lse);

  std::lock_guard<std::mutex> lock(g_mu);
  CopyStreams* cs = nullptr;
  cudaError_t e = copy_streams(&cs);
  if (e != cudaSuccess) return e;
  // the copy streams start after the work already on `stream`
  e = cudaEventRecord(cs->entry, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->in, cs->entry, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->out, cs->entry, 0);
  // the per-row vectors of every row, once
  if (e == cudaSuccess) e = cudaMemcpyAsync(td, t_host, N * 4, cudaMemcpyHostToDevice, cs->in);
  if (e == cudaSuccess) e = cudaMemcpyAsync(gd, g_host, N * 4, cudaMemcpyHostToDevice, cs->in);
  if (e == cudaSuccess && md != nullptr)
    e = cudaMemcpyAsync(md, mask_host, N, cudaMemcpyHostToDevice, cs->in);
  if (e != cudaSuccess) return e;

  // rows of `ld` elements -> dense rows, or back; one plain copy when dense
  auto rows_copy = [&](void* dst, size_t dpitch, const void* src, size_t spitch, int64_t n,
                       cudaMemcpyKind kind, cudaStream_t s) {
    if (dpitch == row_bytes && spitch == row_bytes)
      return cudaMemcpyAsync(dst, src, row_bytes * n, kind, s);
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, row_bytes, static_cast<size_t>(n), kind, s);
  };
  const char* xh = static_cast<const char*>(x_host);
  char* gxh = static_cast<char*>(gx_host);
  const size_t xpitch = static_cast<size_t>(ld) * esize, gpitch = static_cast<size_t>(ld_grad) * esize;
  int64_t r0 = 0;
  for (int64_t k = 0; k < chunks && e == cudaSuccess; r0 += plan[k], ++k) {
    const int s = static_cast<int>(k % kHostSlots);
    const int64_t n = plan[k];
    char* xd = w + L.slots + static_cast<size_t>(s) * L.slot_bytes;
    char* gxd = xd + L.slot_gx;

    // copy in, once the slot's previous chunk has been copied out
    if (k >= kHostSlots) e = cudaStreamWaitEvent(cs->in, cs->out_done[s], 0);
    if (e == cudaSuccess)
      e = rows_copy(xd, row_bytes, xh + r0 * xpitch, xpitch, n, cudaMemcpyHostToDevice, cs->in);
    if (e == cudaSuccess) e = cudaEventRecord(cs->in_done[s], cs->in);
    // compute on the caller's stream
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, cs->in_done[s], 0);
    if (e == cudaSuccess)
      e = launch_forward_backward(xd, dtype, n, V, V, td + r0, md != nullptr ? md + r0 : nullptr,
                                  T, gd + r0, lpd + r0, lsed + r0, gxd, V, err, stream);
    if (e == cudaSuccess) e = cudaEventRecord(cs->cmp_done[s], stream);
    // copy out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->out, cs->cmp_done[s], 0);
    if (e == cudaSuccess)
      e = rows_copy(gxh + r0 * gpitch, gpitch, gxd, row_bytes, n, cudaMemcpyDeviceToHost, cs->out);
    if (e == cudaSuccess) e = cudaEventRecord(cs->out_done[s], cs->out);
  }
  // logprob and lse of every row, once (the out-stream has waited for the
  // last chunk's compute), then `stream` continues once all is on the host
  if (e == cudaSuccess) e = cudaMemcpyAsync(lp_host, lpd, N * 4, cudaMemcpyDeviceToHost, cs->out);
  if (e == cudaSuccess) e = cudaMemcpyAsync(lse_host, lsed, N * 4, cudaMemcpyDeviceToHost, cs->out);
  if (e == cudaSuccess) e = cudaEventRecord(cs->done, cs->out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, cs->done, 0);
  return e;
}

}  // namespace slp
