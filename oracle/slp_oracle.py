"""fp64 CPU oracle for selected-token log-probabilities.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it.  It shares no code, constant or helper with
the CUDA library; the only thing the two sides share is the seeded input
generator, which holds none of the method's arithmetic.

What it computes (the plain definition, written out in float64):

    z[n, v]   = x[n, v] / T
    lse[n]    = max_v z[n, v] + log( sum_v exp(z[n, v] - max_v z[n, v]) )
    logprob[n]= z[n, t_n] - lse[n]                       (= -cross_entropy(z, t) at
                                                          label smoothing 0)
    grad_x[n, v] = g[n] * (1[v == t_n] - exp(z[n, v] - lse[n])) / T

Rows with loss_mask == 0 give logprob = lse = 0 and an all-zero gradient.

Sources (page title, then the section):
  * Megatron-LM issue #6700 "Avoid full-vocabulary TP gather for selected-token
    logprobs", section "Proposed solution": the identity
    log_softmax(logits)[target] == -cross_entropy(logits, target) at label
    smoothing 0, and numerically stable normalisation.
  * torchforge PR #608 "Reduce reference model memory with parallel logprob
    computation", section "Implementation": the log-sum-exp trick (max, then sum
    of exp(x - max)), and the target logit gathered once.
  * NeMo-RL PR #4222 "chunk target logprobs without tensor parallelism", section
    "Changes": backward writes (onehot - softmax) * grad_output into a buffer of
    the logits' dtype, recomputing the softmax from the saved inputs.
  * verl PR #7733 "memory-efficient chunked top-k KL", section "Design & Code
    Changes": the per-token fp32 logZ is what the forward keeps for backward.
  * slime issue #2253 "full-vocab fp32 logits over the packed sequence -> OOM",
    maintainer analysis: only loss_mask == 1 rows are computed, before the
    vocabulary projection; off-mask values are zero after the scatter.

Readings where the pages are silent (each is also listed in the design notes):
  * temperature divides the logits before the softmax (z = x / T); the gradient
    is taken with respect to the raw logits, so it carries the factor 1/T;
  * lse is the log-sum-exp of the scaled logits z;
  * an all -inf row gives NaN (as log_softmax does); a target on a -inf column
    gives logprob = -inf;
  * the LM head has no bias; its logits are h @ W^T in float64.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, invariants, finite differences and independent library routines.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "decode_bf16",
    "selected_logprob_forward",
    "selected_logprob_backward",
    "lmhead_logits",
    "lmhead_forward",
    "lmhead_backward",
    "lmhead_dh_rows",
    "lmhead_dW_rows",
    "entropy_forward",
    "entropy_backward",
    "topk_kl_forward",
    "topk_kl_backward",
]


def decode_bf16(bits) -> np.ndarray:
    """Exact float64 values of bfloat16 numbers given as their 16-bit patterns.

    A bfloat16 is the upper half of an IEEE binary32, so widening is a 16-bit
    left shift of the pattern: no rounding is involved.
    """
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def _as_f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def _active_rows(N: int, mask) -> np.ndarray:
    if mask is None:
        return np.ones(N, dtype=bool)
    return np.asarray(mask).reshape(N) != 0


def selected_logprob_forward(x, t, mask, T: float):
    """Forward of the selected-token log-probability for every row.

    x: [N, V] real logits (any float dtype; widened to float64).
    t: [N] integer targets in [0, V).  mask: [N] (nonzero = compute) or None.
    T: temperature > 0.

    Returns (logprob[N], lse[N]) in float64; inactive rows are 0.

    Follows torchforge PR #608, "Implementation" (max, sum of exp(x - max),
    target logit), on the scaled logits x / T; the identity with
    -cross_entropy is Megatron-LM issue #6700, "Proposed solution".
    """
    x = _as_f64(x)
    N = x.shape[0]
    t = np.asarray(t).reshape(N).astype(np.int64)
    active = _active_rows(N, mask)
    logprob = np.zeros(N, dtype=np.float64)
    lse = np.zeros(N, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        for n in range(N):
            if not active[n]:
                continue
            z = x[n] / T
            M = np.max(z)
            S = np.sum(np.exp(z - M))
            lse[n] = M + np.log(S)
            logprob[n] = z[t[n]] - lse[n]
    return logprob, lse


def selected_logprob_backward(x, t, mask, T: float, lse, grad_out):
    """Gradient of sum_n grad_out[n] * logprob[n] with respect to the raw logits.

    grad_x[n, v] = grad_out[n] * (1[v == t_n] - exp(x[n, v] / T - lse[n])) / T,
    with the softmax recomputed from x and the saved lse (NeMo-RL PR #4222,
    "Changes": (onehot - softmax) * grad_output; verl PR #7733, "Design & Code
    Changes": recompute from the saved per-token logZ).  Inactive rows are 0.
    """
    x = _as_f64(x)
    N, V = x.shape
    t = np.asarray(t).reshape(N).astype(np.int64)
    lse = _as_f64(lse).reshape(N)
    g = _as_f64(grad_out).reshape(N)
    active = _active_rows(N, mask)
    grad = np.zeros((N, V), dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        for n in range(N):
            if not active[n]:
                continue
            p = np.exp(x[n] / T - lse[n])
            onehot = np.zeros(V, dtype=np.float64)
            onehot[t[n]] = 1.0
            grad[n] = g[n] * (onehot - p) / T
    return grad


def lmhead_logits(h, W) -> np.ndarray:
    """LM-head logits h @ W^T in float64 (no bias).

    h: [N, d], W: [V, d].  The products of two bfloat16 values are exact in
    float64, so only the summation order is left to the library matmul.
    """
    return _as_f64(h) @ _as_f64(W).T


def lmhead_forward(h, W, t, mask, T: float):
    """Selected-token log-probabilities through the LM head.

    Only rows with mask != 0 are projected to the vocabulary (slime issue
    #2253, maintainer analysis: keep trainable rows before the vocabulary
    projection, compute compact rows, scatter scalars back); the others return
    logprob = lse = 0.
    """
    h = _as_f64(h)
    N = h.shape[0]
    active = _active_rows(N, mask)
    t = np.asarray(t).reshape(N).astype(np.int64)
    logprob = np.zeros(N, dtype=np.float64)
    lse = np.zeros(N, dtype=np.float64)
    rows = np.nonzero(active)[0]
    if rows.size:
        x = lmhead_logits(h[rows], W)
        lp_c, lse_c = selected_logprob_forward(x, t[rows], None, T)
        logprob[rows] = lp_c
        lse[rows] = lse_c
    return logprob, lse


def lmhead_backward(h, W, t, mask, T: float, lse, grad_out):
    """Gradients of sum_n grad_out[n] * logprob[n] with respect to h and W.

    dz = selected_logprob_backward of the compact logits; then
    dh = dz @ W and dW = dz^T @ h over the active rows only.  Inactive rows of
    dh are 0 (Megatron-LM issue #6700, "Prototype correctness": masked
    positions have exactly zero gradient).
    Returns (dh [N, d], dW [V, d]) in float64.
    """
    h = _as_f64(h)
    W = _as_f64(W)
    N, d = h.shape
    V = W.shape[0]
    active = _active_rows(N, mask)
    t = np.asarray(t).reshape(N).astype(np.int64)
    lse = _as_f64(lse).reshape(N)
    g = _as_f64(grad_out).reshape(N)
    dh = np.zeros((N, d), dtype=np.float64)
    dW = np.zeros((V, d), dtype=np.float64)
    rows = np.nonzero(active)[0]
    if rows.size:
        x = lmhead_logits(h[rows], W)
        dz = selected_logprob_backward(x, t[rows], None, T, lse[rows], g[rows])
        dh[rows] = dz @ W
        dW = dz.T @ h[rows]
    return dh, dW


def lmhead_dh_rows(h, W, t, mask, T: float, lse, grad_out, rows):
    """Rows `rows` of dh from lmhead_backward: for an active row n,
    dh[n] = dz[n] @ W with dz[n, v] = g_n (1[v = t_n] - exp(h_n.W_v / T -
    lse_n)) / T; an inactive row is 0.  Needs only the requested rows' own
    lse.  The requested active rows are projected together, as one smaller
    instance of lmhead_backward's products."""
    W = _as_f64(W)
    h = _as_f64(h)
    N = h.shape[0]
    active = _active_rows(N, mask)
    t = np.asarray(t).reshape(N).astype(np.int64)
    lse = _as_f64(lse).reshape(N)
    g = _as_f64(grad_out).reshape(N)
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    out = np.zeros((rows.size, W.shape[1]), dtype=np.float64)
    sel = np.nonzero(active[rows])[0]
    if sel.size:
        r = rows[sel]
        x = lmhead_logits(h[r], W)
        dz = selected_logprob_backward(x, t[r], None, T, lse[r], g[r])
        out[sel] = dz @ W
    return out


def lmhead_dW_rows(h, W, t, mask, T: float, lse, grad_out, vrows):
    """Rows `vrows` of dW from lmhead_backward: dW[v] = sum over active rows n
    of dz[n, v] h[n], with dz[n, v] = g_n (1[v = t_n] - exp(h_n.W_v / T -
    lse_n)) / T.  Needs lse of every active row (from lmhead_forward)."""
    h = _as_f64(h)
    W = _as_f64(W)
    N = h.shape[0]
    active = _active_rows(N, mask)
    rows = np.nonzero(active)[0]
    t = np.asarray(t).reshape(N).astype(np.int64)[rows]
    lse = _as_f64(lse).reshape(N)[rows]
    g = _as_f64(grad_out).reshape(N)[rows]
    hr = h[rows]
    out = np.zeros((len(vrows), h.shape[1]), dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        for k, v in enumerate(vrows):
            z = hr @ W[v] / T
            dz = g * ((t == v).astype(np.float64) - np.exp(z - lse)) / T
            out[k] = dz @ hr
    return out


def entropy_forward(x, t, mask, T: float):
    """Selected-token log-probability, lse and the per-token entropy of the
    same softmax, H[n] = -sum_v p[n, v] log p[n, v] with p = softmax(x[n] / T)
    (slime issue #2253: get_log_probs_and_entropy computes both over the same
    rows).  Returns (logprob, lse, entropy) in float64; inactive rows are 0."""
    x = _as_f64(x)
    N = x.shape[0]
    lp, lse = selected_logprob_forward(x, t, mask, T)
    active = _active_rows(N, mask)
    H = np.zeros(N, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        for n in range(N):
            if not active[n]:
                continue
            logp = x[n] / T - lse[n]
            p = np.exp(logp)
            H[n] = -np.sum(np.where(p > 0, p * logp, 0.0))
    return lp, lse, H


def entropy_backward(x, t, mask, T: float, lse, H, grad_out, grad_entropy):
    """Gradient of sum_n (g[n] logprob[n] + gH[n] H[n]) with respect to x:
    g (1[v = t] - p_v) / T - gH p_v (log p_v + H) / T, using
    dH/dz_v = -p_v (log p_v + H) for z = x / T."""
    x = _as_f64(x)
    N, V = x.shape
    grad = selected_logprob_backward(x, t, mask, T, lse, grad_out)
    active = _active_rows(N, mask)
    lse = _as_f64(lse).reshape(N)
    H = _as_f64(H).reshape(N)
    gH = _as_f64(grad_entropy).reshape(N)
    with np.errstate(invalid="ignore", over="ignore"):
        for n in range(N):
            if not active[n]:
                continue
            logp = x[n] / T - lse[n]
            p = np.exp(logp)
            grad[n] -= gH[n] * np.where(p > 0, p * (logp + H[n]), 0.0) / T
    return grad


def topk_kl_forward(x, ids, teacher_logp, mask, T: float, clamp_min=None):
    """Forward KL of the student softmax(x / T) against a teacher given only by
    its top-K token ids and log-probabilities, over that support (verl PR
    #7733 "memory-efficient chunked top-k KL", "Design & Code Changes":
    gather the teacher top-k plus the student statistics at those ids, with
    the student's global logZ):

        ls[k] = x[n, ids[n, k]] / T - lse[n]         (student log-prob)
        lc[k] = max(ls[k], clamp_min)                 (when a clamp is given)
        kl[n] = sum_k exp(lt[k]) (lt[k] - lc[k])
        student_mass[n] = sum_k exp(ls[k]),  teacher_mass[n] = sum_k exp(lt[k])

    Returns (kl, student_mass, teacher_mass, lse) in float64; inactive rows 0.
    """
    x = _as_f64(x)
    N = x.shape[0]
    ids = np.asarray(ids).reshape(N, -1).astype(np.int64)
    lt = _as_f64(teacher_logp).reshape(N, -1)
    active = _active_rows(N, mask)
    _, lse = selected_logprob_forward(x, np.zeros(N, np.int64), mask, T)
    kl = np.zeros(N)
    sm = np.zeros(N)
    tm = np.zeros(N)
    for n in range(N):
        if not active[n]:
            continue
        ls = x[n, ids[n]] / T - lse[n]
        lc = ls if clamp_min is None else np.maximum(ls, clamp_min)
        p = np.exp(lt[n])
        kl[n] = np.sum(p * (lt[n] - lc))
        sm[n] = np.sum(np.exp(ls))
        tm[n] = np.sum(p)
    return kl, sm, tm, lse


def topk_kl_backward(x, ids, teacher_logp, mask, T: float, clamp_min, lse, grad_kl):
    """Gradient of sum_n g[n] kl[n] with respect to x.  d kl / d ls[k] is
    -p[k] where ls[k] >= clamp_min (the clamp's flat side gives 0), and
    d ls[k] / d x[v] = (1[v = ids[k]] - q[v]) / T with q = softmax(x / T):

        grad_x[n, v] = g[n] / T * ( P q[v] - sum_{k: ids[k] = v, kept} p[k] ),
        P = sum of p[k] over the kept k.
    """
    x = _as_f64(x)
    N, V = x.shape
    ids = np.asarray(ids).reshape(N, -1).astype(np.int64)
    lt = _as_f64(teacher_logp).reshape(N, -1)
    lse = _as_f64(lse).reshape(N)
    g = _as_f64(grad_kl).reshape(N)
    active = _active_rows(N, mask)
    grad = np.zeros((N, V))
    for n in range(N):
        if not active[n]:
            continue
        ls = x[n, ids[n]] / T - lse[n]
        keep = np.ones_like(ls, bool) if clamp_min is None else ls >= clamp_min
        p = np.exp(lt[n]) * keep
        q = np.exp(x[n] / T - lse[n])
        row = p.sum() * q
        np.add.at(row, ids[n], -p)
        grad[n] = g[n] * row / T
    return grad
