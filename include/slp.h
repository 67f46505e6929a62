/*
 * slp.h - selected-token log-probabilities over a large vocabulary, on one
 * NVIDIA GB300 (sm_103a).  C ABI of libslp.so.
 *
 * For every row n of a logits matrix x[N, V], with target token t[n] and
 * temperature T:
 *
 *     logprob[n] = x[n, t_n] / T - logsumexp_v( x[n, v] / T )
 *     lse[n]     = logsumexp_v( x[n, v] / T )
 *
 * which is -cross_entropy(x / T, t) at label smoothing 0 (Megatron-LM issue
 * #6700 "Avoid full-vocabulary TP gather for selected-token logprobs",
 * "Proposed solution").  The backward pass writes
 *
 *     grad_x[n, v] = grad_out[n] * (1[v == t_n] - exp(x[n, v] / T - lse[n])) / T
 *
 * recomputing the softmax from x and the saved lse instead of keeping a float32
 * [N, V] buffer (NeMo-RL PR #4222 "chunk target logprobs without tensor
 * parallelism", "Changes"; verl PR #7733 "memory-efficient chunked top-k KL",
 * "Design & Code Changes").  A second pair of calls fuses the LM-head
 * projection x = h W^T with the same log-sum-exp, computing only rows whose
 * loss mask is 1 (slime issue #2253 "full-vocab fp32 logits over the packed
 * sequence -> OOM", maintainer analysis), so the logits are never stored.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All array arguments are DEVICE pointers on the current CUDA device,
 *    allocated and owned by the caller (except the *_host buffers of
 *    slp_forward_backward_host, which are page-locked host memory).  The library allocates no device
 *    memory, keeps no pointer after a call returns and never synchronises:
 *    every kernel is enqueued on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream), so results are ready when the stream
 *    reaches that point.  The calls contain no host-device synchronisation and
 *    no allocation, so they may be captured in a CUDA graph.
 *  - Matrices are row-major.  `ld` is the row stride in elements (ld >= V).
 *  - Outputs are overwritten, never accumulated into (except the fp32 dW of
 *    slp_lmhead_backward_accumulate), and must not overlap any input: in
 *    particular grad_x may not share memory with x (the target's element
 *    is recomputed from x after the row's gradient has been stored).
 *  - `mask` is optional (NULL = every row active).  mask[n] == 0 makes row n
 *    inactive: its logprob and lse are +0.0 and its gradient row is +0.0,
 *    bit for bit (Megatron-LM issue #6700, "Prototype correctness": masked
 *    positions have exactly zero gradient).
 *  - Argument errors are reported synchronously by the return value, before
 *    anything is launched.  N == 0 is a successful no-op.
 *  - Data errors are found on the device: a target outside [0, V) on an
 *    active row ORs SLP_DATA_ERR_TARGET into *err (when err is not NULL) and
 *    makes that row's outputs NaN.  No kernel traps or asserts.
 *  - All offsets are 64-bit (N * ld may exceed 2^32).
 */
#ifndef SLP_H_
#define SLP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the logits (and of their gradient). */
typedef enum { SLP_BF16 = 0, SLP_F32 = 1 } slp_dtype;

/* Return values. */
typedef enum {
  SLP_OK = 0,
  SLP_ERR_INVALID_ARG = 1, /* NULL required pointer, N < 0, V <= 0, ld < V,
                              T not finite or <= 0, unknown dtype, ...      */
  SLP_ERR_UNSUPPORTED = 2, /* shape the kernels do not handle (see per call) */
  SLP_ERR_MISALIGNED = 3,  /* pointer/stride alignment the call requires    */
  SLP_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than required       */
  SLP_ERR_CUDA = 5         /* a CUDA runtime call or launch failed          */
} slp_status;

/* Bits OR-ed into the optional device error word. */
#define SLP_DATA_ERR_TARGET 1    /* target outside [0, V) on an active row          */
#define SLP_DEVICE_ERR_TIMEOUT 2 /* a pipeline wait inside an LM-head kernel gave up
                                    after its bound (two seconds unless
                                    slp_lmhead_set_wait_limit_ns set another); that
                                    call's outputs are undefined (the kernel drained
                                    its copies and tensor-core work and returned
                                    instead of hanging) */
#define SLP_DEVICE_ERR_BOUNDS 4  /* only in a library built with -DSLP_DEBUG_BOUNDS: a
                                    kernel refused a global access outside every buffer
                                    its call was given (the access was skipped)     */

/*
 * slp_forward - selected-token log-probability and row log-sum-exp.
 *
 * Defined by: Megatron-LM issue #6700, "Proposed solution" (the identity with
 * -cross_entropy, stable normalisation); torchforge PR #608 "Reduce reference
 * model memory with parallel logprob computation", "Implementation" (max,
 * sum of exp(x - max), target gather); NeMo-RL PR #4222, "Changes" (fp32
 * log-sum-exp over low-precision logits that are never upcast as a whole).
 *
 *   x        [N, ld] logits of type `dtype` (bf16 or f32); columns >= V unread.
 *   dtype    SLP_BF16 or SLP_F32.
 *   N, V, ld rows, vocabulary size, row stride in elements (ld >= V).
 *   t        [N] int32 targets.
 *   mask     [N] uint8 loss mask or NULL.
 *   T        temperature, finite and > 0.
 *   logprob  [N] float32 out.
 *   lse      [N] float32 out: log-sum-exp of x / T (kept for slp_backward).
 *   err      optional int32 device error word (only ever OR-ed into).
 *   stream   cudaStream_t.
 *
 * Any ld and alignment is accepted; rows whose base address is 16-byte
 * aligned (x aligned and ld * sizeof(element) a multiple of 16) take the
 * 128-bit vector path.  An all -inf row gives NaN; a target on a -inf column
 * gives logprob = -inf.
 */
int slp_forward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                const int32_t* t, const uint8_t* mask, float T,
                float* logprob, float* lse, int32_t* err, void* stream);

/*
 * slp_backward - gradient of sum_n grad_out[n] * logprob[n] w.r.t. x.
 *
 * Defined by: NeMo-RL PR #4222, "Changes" ((onehot - softmax) * grad_output
 * written into a buffer of the logits' dtype, softmax recomputed); verl PR
 * #7733, "Design & Code Changes" (recompute from the saved per-token fp32
 * logZ).  The factor 1/T is the derivative of x / T.
 *
 *   x, dtype, N, V, ld, t, mask, T   as for slp_forward (same values).
 *   lse       [N] float32, as returned by slp_forward.
 *   grad_out  [N] float32 upstream gradient of logprob.
 *   grad_x    [N, ld_grad] out, same element type as x; columns >= V are not
 *             written.  Float32 arithmetic, rounded to nearest-even into bf16.
 *   ld_grad   row stride of grad_x in elements (>= V).
 *   err       optional device error word.
 */
int slp_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                 const int32_t* t, const uint8_t* mask, float T,
                 const float* lse, const float* grad_out,
                 void* grad_x, int64_t ld_grad, int32_t* err, void* stream);

/*
 * slp_forward_entropy - slp_forward plus the per-token entropy of the same
 * softmax, H[n] = -sum_v p[n,v] log p[n,v] with p = softmax(x[n] / T), from
 * the same single read of the logits (one more running accumulator).
 *
 * Defined by: slime issue #2253 (get_log_probs_and_entropy computes the
 * selected log-probability and the entropy over the same rows); the entropy
 * itself is the textbook definition.
 *
 *   as slp_forward, plus entropy [N] float32 out (0 on inactive rows, NaN
 *   where logprob is NaN).
 */
int slp_forward_entropy(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                        const int32_t* t, const uint8_t* mask, float T,
                        float* logprob, float* lse, float* entropy, int32_t* err, void* stream);

/*
 * slp_backward_entropy - gradient of sum_n (g[n] logprob[n] + gH[n] H[n])
 * with respect to x:
 *
 *   grad_x[n,v] = ( g[n] (1[v == t_n] - p_v) - gH[n] p_v (log p_v + H[n]) ) / T
 *
 * (dH/dz_v = -p_v (log p_v + H) for z = x / T), recomputing p from x and lse.
 *
 *   as slp_backward, plus entropy [N] from slp_forward_entropy and
 *   grad_entropy [N] float32.  grad_out or grad_entropy may be NULL, meaning
 *   zero.
 */
int slp_backward_entropy(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                         const int32_t* t, const uint8_t* mask, float T,
                         const float* lse, const float* entropy,
                         const float* grad_out, const float* grad_entropy,
                         void* grad_x, int64_t ld_grad, int32_t* err, void* stream);

/*
 * slp_topk_kl_forward - per-token forward KL of the student softmax(x / T)
 * against a teacher given only by its top-K token ids and log-probabilities,
 * over that support, with the student's full-vocabulary logZ.
 *
 * Defined by: verl PR #7733 "memory-efficient chunked top-k KL", "What does
 * this PR do?" and "Design & Code Changes" (teacher top-k plus student
 * statistics, global logZ from MAX/SUM reductions, recompute in backward):
 *
 *   ls[k] = x[n, ids[n,k]] / T - lse[n],   lc[k] = max(ls[k], clamp_min)
 *   kl[n] = sum_k exp(lt[n,k]) (lt[n,k] - lc[k])
 *   student_mass[n] = sum_k exp(ls[k]),   teacher_mass[n] = sum_k exp(lt[n,k])
 *
 *   x, dtype, N, V, ld, mask, T, err, stream   as for slp_forward.
 *   ids           [N, K] int32 teacher token ids, row-major (repeats allowed).
 *   teacher_logp  [N, K] float32 teacher log-probabilities of those ids.
 *   K             entries per row, >= 1.
 *   clamp_min     lower clamp of the student log-probabilities in kl
 *                 (-INFINITY for none; the pages' runs use -10).
 *   kl, student_mass, teacher_mass, lse   [N] float32 out (0 on inactive rows).
 * An id outside [0, V) on an active row sets SLP_DATA_ERR_TARGET and makes
 * that row's outputs NaN.
 */
int slp_topk_kl_forward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                        const int32_t* ids, const float* teacher_logp, int64_t K,
                        const uint8_t* mask, float T, float clamp_min,
                        float* kl, float* student_mass, float* teacher_mass, float* lse,
                        int32_t* err, void* stream);

/*
 * slp_topk_kl_backward - gradient of sum_n grad_kl[n] kl[n] with respect to x:
 *
 *   grad_x[n,v] = grad_kl[n] / T * ( P q[v] - sum_{k: ids[k] = v, ls[k] >= clamp_min}
 *                 exp(lt[k]) ),   P = sum of exp(lt[k]) over the kept k,
 *
 * with q = softmax(x / T) recomputed from x and the saved lse (the clamp's
 * flat side contributes no gradient).  Arguments as slp_topk_kl_forward plus
 * lse (from it), grad_kl [N] float32, grad_x [N, ld_grad] in x's dtype.
 * Returns SLP_ERR_UNSUPPORTED for K above 16384 (the teacher entries are
 * staged in shared memory).
 */
int slp_topk_kl_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                         const int32_t* ids, const float* teacher_logp, int64_t K,
                         const uint8_t* mask, float T, float clamp_min, const float* lse,
                         const float* grad_kl, void* grad_x, int64_t ld_grad,
                         int32_t* err, void* stream);

/*
 * slp_forward_backward - slp_forward and slp_backward in one pass, for the
 * training case where grad_out is known when the forward runs (for example
 * g = -advantage for a plain policy-gradient loss).
 *
 * Defined by: the two calls above (same definitions, same results within
 * their tolerances).  Each row is read from HBM once and kept on chip
 * between the log-sum-exp and the gradient pass: a row of at most 32 KB by
 * one warp (registers plus a shared-memory slot), a longer one by a
 * thread-block cluster that splits it across up to 8 CTAs' registers and
 * shared memory (and, for long float32 rows, tensor memory as well, 64 KB
 * per CTA).  So the row's bytes are read once
 * instead of twice (NeMo-RL PR #4222, "Changes": recompute the softmax rather
 * than store it).  Rows that are not 16-byte aligned, or longer than eight
 * such CTAs hold (about 1.1 MB), are served by slp_forward followed by
 * slp_backward.
 *
 *   x, dtype, N, V, ld, t, mask, T   as for slp_forward.
 *   grad_out  [N] float32 upstream gradient of logprob.
 *   logprob, lse  [N] float32 out, as from slp_forward.
 *   grad_x, ld_grad, err, stream     as for slp_backward.
 */
int slp_forward_backward(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                         const int32_t* t, const uint8_t* mask, float T,
                         const float* grad_out, float* logprob, float* lse,
                         void* grad_x, int64_t ld_grad, int32_t* err, void* stream);

/*
 * slp_forward_backward_entropy - slp_forward_entropy and slp_backward_entropy
 * in one pass, for a loss whose per-token weights are known when the forward
 * runs: sum_n g[n] logprob[n] + gH[n] H[n] (for example a policy-gradient
 * term with an entropy bonus, gH = -beta).
 *
 * Defined by: the two entropy calls above (same definitions, same results
 * within their tolerances).  The row is kept on chip as in
 * slp_forward_backward, so it is read from HBM once instead of twice.  The
 * gradient is computed from the lse and entropy this call writes, with the
 * same per-element arithmetic as slp_backward_entropy.  Rows that are not
 * 16-byte aligned, or longer than about 1.1 MB, are served by
 * slp_forward_entropy followed by slp_backward_entropy.
 *
 *   x, dtype, N, V, ld, t, mask, T   as for slp_forward.
 *   grad_out, grad_entropy  [N] float32 upstream gradients of logprob and of
 *                  the entropy; either may be NULL, meaning zero.
 *   logprob, lse, entropy  [N] float32 out, as from slp_forward_entropy.
 *   grad_x, ld_grad, err, stream     as for slp_backward.
 */
int slp_forward_backward_entropy(const void* x, int dtype, int64_t N, int64_t V, int64_t ld,
                                 const int32_t* t, const uint8_t* mask, float T,
                                 const float* grad_out, const float* grad_entropy, float* logprob,
                                 float* lse, float* entropy, void* grad_x, int64_t ld_grad,
                                 int32_t* err, void* stream);

/*
 * slp_forward_backward_host - slp_forward_backward for logits that live in
 * pinned host memory (for example after an offload), streamed through the GPU
 * in row chunks.  No counterpart in the pages: it only moves the rows of the
 * call above to and from the host.
 *
 * Three streams overlap: chunk k+1 is copied in while chunk k is computed on
 * `stream` and chunk k-1's results are copied out.  The copy streams are the
 * library's own (created once per device).  They wait for `stream` at entry,
 * and `stream` waits for the last copy before the call returns.  Work enqueued
 * on `stream` after the call therefore sees the results in host memory,
 * which are complete once `stream` has reached that point.  The call does
 * not synchronise.
 *
 *   x_host   [N, ld] rows of dtype in page-locked host memory (cudaHostAlloc
 *            or cudaHostRegister); t_host [N] int32, mask_host [N] uint8
 *            (nullable), g_host [N] float32: page-locked too.
 *   logprob_host, lse_host [N] float32 and grad_x_host [N, ld_grad] (dtype)
 *            out, page-locked.
 *   rows_per_chunk  rows per chunk; 0 picks about 64 MB of logits per chunk.
 *   ws, ws_bytes  device workspace of at least
 *            slp_forward_backward_host_workspace_size(N, V, dtype,
 *            rows_per_chunk) bytes, 256-byte aligned.
 *   err, stream  as for slp_backward (err is a device pointer).
 * Returns SLP_ERR_INVALID_ARG if a host buffer is not page-locked, and
 * SLP_ERR_WORKSPACE if ws is too small.
 */
size_t slp_forward_backward_host_workspace_size(int64_t N, int64_t V, int dtype,
                                                int64_t rows_per_chunk);
int slp_forward_backward_host(const void* x_host, int dtype, int64_t N, int64_t V, int64_t ld,
                              const int32_t* t_host, const uint8_t* mask_host, float T,
                              const float* g_host, float* logprob_host, float* lse_host,
                              void* grad_x_host, int64_t ld_grad, int64_t rows_per_chunk,
                              void* ws, size_t ws_bytes, int32_t* err, void* stream);

/*
 * slp_lmhead_workspace_size - the recommended device workspace of
 * slp_lmhead_backward for these sizes (enough for slp_lmhead_forward too):
 * the backward then runs in vocabulary chunks of 65536 columns.  Returns 0
 * for invalid sizes.
 *
 * slp_lmhead_workspace_size_min - the least workspace slp_lmhead_backward
 * accepts: chunks of 16384 columns, a quarter of the default dz buffer and
 * fewer split-K partials, for more GEMM launches.  Between the two, the
 * backward uses the widest chunk that fits (65536, 32768 or 16384 columns).
 *
 * slp_lmhead_forward_workspace_size - the smaller amount slp_lmhead_forward
 * alone needs (compacted hidden rows and per-slab log-sum-exp partials).
 *
 * The backward workspace holds the compacted rows, a bf16 dz buffer of
 * roundup(N,256) x chunk elements, float32 split-K partials of dh and a
 * float32 dh accumulator.  Workspaces of different chunk widths give results
 * that agree within the LM-head tolerances, not bit for bit: the dh sums are
 * regrouped.
 */
size_t slp_lmhead_workspace_size(int64_t N, int64_t V, int64_t d);
size_t slp_lmhead_workspace_size_min(int64_t N, int64_t V, int64_t d);
size_t slp_lmhead_forward_workspace_size(int64_t N, int64_t V, int64_t d);

/*
 * slp_lmhead_workspace_size_max - bytes of workspace with which the LM-head
 * backward runs the whole vocabulary as one chunk.  Given a larger workspace
 * than slp_lmhead_workspace_size, the backward uses the widest chunk that fits:
 * the whole vocabulary, else 131072 columns, else 65536.  Fewer chunks mean
 * fewer GEMM launches.  At N=8192, V=151936, d=2560 this takes 3.96 GB
 * instead of 1.86 GB and is about 2 % faster.  Results agree within the
 * LM-head tolerances, not bit for bit: the dh sums are regrouped.  Returns 0
 * for invalid sizes.
 */
size_t slp_lmhead_workspace_size_max(int64_t N, int64_t V, int64_t d);

/*
 * slp_lmhead_forward - selected-token log-probabilities through the LM head,
 * logits never stored.
 *
 * The GEMMs run on pairs of CTAs (thread-block clusters of two, one
 * tcgen05 MMA over both) that claim their tiles from a counter in the
 * workspace; results do not depend on which pair computes which tile.  On a
 * device that cannot co-schedule such pairs, or
 * with SLP_LMHEAD_CTA_PAIRS=0 in the environment before the first LM-head
 * call or workspace query, they run one CTA per tile.  The two forms agree
 * within the LM-head tolerances and need workspaces of different sizes: ask
 * the workspace functions in the same process that makes the calls.
 *
 * Defined by: the slp_forward definition applied to x = h W^T (no bias),
 * computing only rows with mask[n] != 0 before the vocabulary projection and
 * scattering the per-row scalars back (slime issue #2253, maintainer
 * analysis); Megatron-LM issue #6700, "Alternatives considered" (a fused
 * LM-head / cross-entropy kernel).
 *
 *   h        [N, d] bf16 hidden states, row-major, 16-byte aligned.
 *   W        [V, d] bf16 output embedding, row-major, 16-byte aligned.
 *   N, V, d  d must be a positive multiple of 64.
 *   t, mask, T, logprob, lse, err, stream   as for slp_forward.  The logits
 *            are accumulated in float32 and not rounded before the
 *            log-sum-exp.
 *   ws, ws_bytes  device workspace of at least
 *            slp_lmhead_forward_workspace_size(N, V, d) bytes, 256-byte
 *            aligned; its contents on entry do not matter.
 */
int slp_lmhead_forward(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                       const int32_t* t, const uint8_t* mask, float T,
                       float* logprob, float* lse,
                       void* ws, size_t ws_bytes, int32_t* err, void* stream);

/*
 * slp_lmhead_backward - gradients of sum_n grad_out[n] * logprob[n] with
 * respect to h and W for the fused LM head.
 *
 *   dz[n, v] = grad_out[n] * (1[v == t_n] - exp(z[n, v] - lse[n])) / T with
 *   z = h W^T / T recomputed from the saved lse (as for slp_backward);
 *   dh = dz W and dW = dz^T h over the active rows, float32 accumulation,
 *   rounded to nearest-even into bf16.  Inactive rows of dh are +0.0.
 *
 *   h, W, N, V, d, t, mask, T   as for slp_lmhead_forward (same values).
 *   lse       [N] float32 from slp_lmhead_forward.
 *   grad_out  [N] float32.
 *   dh        [N, d] bf16 out.      dW  [V, d] bf16 out (overwritten).
 *   ws, ws_bytes  at least slp_lmhead_workspace_size_min(N, V, d) bytes
 *             (slp_lmhead_workspace_size recommended), 256-byte aligned;
 *             contents on entry do not matter.  The chunk width follows
 *             ws_bytes (see slp_lmhead_workspace_size).
 *   err, stream   as for slp_lmhead_forward.
 * A row whose target is outside [0, V) is flagged in *err, gets a NaN dh row
 * and contributes nothing to dW.
 */
int slp_lmhead_backward(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                        const int32_t* t, const uint8_t* mask, float T,
                        const float* lse, const float* grad_out,
                        void* dh, void* dW,
                        void* ws, size_t ws_bytes, int32_t* err, void* stream);

/*
 * slp_lmhead_forward_noalloc - slp_lmhead_forward without a caller workspace.
 *
 * The source pages have no counterpart to this call; it exists for callers
 * that cannot allocate device memory on demand: their framework owns every
 * byte of device memory through its own pool or budget, or they call from a
 * place where cudaMalloc (which synchronises the whole device) is not
 * acceptable, so they cannot supply the workspace slp_lmhead_forward needs.
 *
 * Same arguments, results and errors as slp_lmhead_forward, minus ws and
 * ws_bytes.  The scratch is one 16 MiB array inside the library's device
 * image, present on every GPU that loads the library until the process
 * exits.  Sizes whose forward workspace
 * (slp_lmhead_forward_workspace_size(N, V, d)) exceeds 16 MiB are rejected
 * with SLP_ERR_WORKSPACE before anything is launched; at d = 2560 and
 * V = 151936 that allows up to N = 1792 rows.
 *
 * The call allocates nothing.  Its first call on a device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current)
 * and keeps it for the life of the process; make that first call before any
 * stream capture.  A cudaDeviceReset on that device ends the context that
 * address belongs to, so the call must not be used on that device after a
 * reset (unload and reload the library instead).  All calls on a device
 * share the array and leave their contents in it (no part has to start
 * zeroed); calls whose work overlaps on the GPU race on it, so serialise
 * them (for example on one stream).
 */
int slp_lmhead_forward_noalloc(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                               const int32_t* t, const uint8_t* mask, float T,
                               float* logprob, float* lse, int32_t* err, void* stream);

/*
 * slp_lmhead_backward_accumulate - slp_lmhead_backward for gradient
 * accumulation across micro-batches: dh is written as in slp_lmhead_backward,
 * and this micro-batch's dW is ADDED into a float32 accumulator,
 *
 *   dW_accum[V, d] += dz^T h      (float32, no rounding to bf16)
 *
 * so a trainer can sum W's gradient over several micro-batches without a
 * separate [V, d] buffer and add.  Same arguments and errors as
 * slp_lmhead_backward with dW replaced by dW_accum (float32, 16-byte
 * aligned).  Each element gets one add per call, in a fixed order, so the
 * result is deterministic.
 *
 * Defined by: slp_lmhead_backward's gradient, summed over the micro-batches
 * of one update (Megatron-LM issue #6700, "Prototype performance": several
 * micro-batches per update).
 */
int slp_lmhead_backward_accumulate(const void* h, const void* W, int64_t N, int64_t V, int64_t d,
                                   const int32_t* t, const uint8_t* mask, float T,
                                   const float* lse, const float* grad_out, void* dh,
                                   float* dW_accum, void* ws, size_t ws_bytes, int32_t* err,
                                   void* stream);

/*
 * slp_lmhead_set_wait_limit_ns - bound, in nanoseconds, of every pipeline wait
 * inside the LM-head kernels launched after this call (process-wide, all
 * devices); ns == 0 restores the default of two seconds.  Returns the bound
 * that was in force.
 *
 * The pages have no counterpart: they only ask that what is not handled be
 * reported explicitly rather than change results silently (Megatron-LM issue
 * #6700, "Compatibility and fallbacks"; slime issue #2253, maintainer
 * analysis: a fail-closed contract).  Every wait in the LM-head GEMMs (a copy
 * landing in shared memory, tensor-core work finishing, an accumulator being
 * drained) counts SM cycles at two per nanosecond, so it lasts at least this
 * long at any clock.  A wait that runs out sets SLP_DEVICE_ERR_TIMEOUT in
 * *err, lets the CTA wait (with a fixed two-second bound) for the copies and
 * tensor-core operations it has already issued, frees its tensor memory and
 * returns; later calls on the stream run normally.  A short bound is for
 * tests of that path and for callers that want an early watchdog; the
 * default is far above any single launch.  Not synchronised with launches in
 * flight: it applies to launches made after it returns.
 */
uint64_t slp_lmhead_set_wait_limit_ns(uint64_t ns);

/*
 * slp_bounds_check_selftest - shows that a library built with
 * -DSLP_DEBUG_BOUNDS checks its kernels' global accesses.  No page has a
 * counterpart: this build stands in for a memory checker, which this library's
 * tests cannot use.
 *
 * buf: device array of at least 8 floats; err: device error word.  In the
 * checked build one kernel is launched whose table of permitted ranges holds
 * buf[0..4) only; it loads and stores buf[4] (inside the caller's array, so
 * nothing is touched that the caller does not own) and stores 1.0f to buf[0].
 * The access to buf[4] must be refused: SLP_DEVICE_ERR_BOUNDS is ORed into
 * *err, buf[4] is left as it was and buf[0] becomes 1.0f.  In a normal build
 * nothing is launched and SLP_ERR_UNSUPPORTED is returned.
 */
int slp_bounds_check_selftest(float* buf, int32_t* err, void* stream);

/* Static, human-readable text for a slp_status value. */
const char* slp_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SLP_H_ */
