"""Selected-token log-probabilities over a large vocabulary on one GB300.

Thin binding over the C ABI of ``libslp.so`` (``include/slp.h``): the
functions below only check tensor properties, allocate outputs with torch
when the caller passes none, and hand raw device pointers plus the current
CUDA stream to the library.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback.

    logprob[n] = x[n, t_n] / T - logsumexp_v(x[n, v] / T)

Low level (same names and arguments as the C ABI):
    slp_forward, slp_backward, slp_lmhead_workspace_size,
    slp_lmhead_forward, slp_lmhead_backward
Autograd:
    selected_logprob(x, t, mask=None, temperature=1.0)
    lmhead_selected_logprob(h, W, t, mask=None, temperature=1.0)
"""

from __future__ import annotations

import torch

from . import _lib
from ._lib import SlpError

__all__ = [
    "SlpError", "slp_forward", "slp_backward", "slp_forward_backward",
    "slp_forward_entropy", "slp_backward_entropy", "slp_forward_backward_entropy",
    "selected_logprob_and_entropy",
    "slp_topk_kl_forward", "slp_topk_kl_backward",
    "slp_lmhead_workspace_size", "slp_lmhead_workspace_size_min", "slp_lmhead_workspace_size_max",
    "slp_lmhead_forward_workspace_size", "slp_lmhead_forward_noalloc",
    "slp_lmhead_backward_accumulate", "slp_lmhead_set_wait_limit_ns",
    "slp_lmhead_forward", "slp_lmhead_backward", "selected_logprob",
    "lmhead_selected_logprob", "library_path",
]

_DTYPES = {torch.bfloat16: _lib.SLP_BF16, torch.float32: _lib.SLP_F32}


def library_path() -> str:
    _lib.load()
    return _lib.LIB_PATH


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_vec(name, v, N, dtype):
    if v.dim() != 1 or v.shape[0] != N or v.dtype != dtype or not v.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [{N}] {dtype} tensor")
    return v


def _span(t):
    """[first, last) byte address range a strided tensor touches."""
    if t.numel() == 0:
        return (t.data_ptr(), t.data_ptr())
    last = sum((n - 1) * st for n, st in zip(t.shape, t.stride()))
    return (t.data_ptr(), t.data_ptr() + (last + 1) * t.element_size())


def _check_disjoint(out_name, out, *inputs):
    """Outputs may not share memory with inputs (slp.h).  Compares address
    ranges, so it also refuses interleaved views of one buffer."""
    a = _span(out)
    for v in inputs:
        if v is None:
            continue
        b = _span(v)
        if a[0] < b[1] and b[0] < a[1]:
            raise ValueError(f"{out_name} must not overlap the inputs")


def _logits_layout(x):
    if x.dim() != 2 or x.dtype not in _DTYPES:
        raise ValueError("x must be a 2-D bfloat16 or float32 tensor")
    N, V = x.shape
    if N > 0 and V > 0 and x.stride(1) != 1:
        raise ValueError("x must have unit column stride")
    ld = x.stride(0) if N > 1 else max(V, 1)
    return N, V, ld


def _check_grad_x(grad_x, x, N, V):
    """A caller's grad_x: [N, V], x's dtype, unit column stride, rows at least
    V apart (the library writes N rows of V elements at its row stride), and
    no overlap with x.  Returns its row stride."""
    if grad_x.dim() != 2 or tuple(grad_x.shape) != (N, V) or grad_x.dtype != x.dtype:
        raise ValueError(f"grad_x must be an [{N}, {V}] {x.dtype} tensor")
    if N > 0 and V > 0 and grad_x.stride(1) != 1:
        raise ValueError("grad_x must have unit column stride")
    ldg = grad_x.stride(0) if N > 1 else max(V, 1)
    if ldg < V:
        raise ValueError("grad_x rows must not overlap (row stride >= V)")
    _check_disjoint("grad_x", grad_x, x)
    return ldg


def _check_mat(name, v, rows, cols, dtype):
    """A caller's [rows, cols] output written densely by the library."""
    if v.dim() != 2 or tuple(v.shape) != (rows, cols) or v.dtype != dtype or not v.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [{rows}, {cols}] {dtype} tensor")
    return v


def _err_ptr(err):
    """The optional device error word: an int32 tensor of at least one
    element (the library ORs status bits into its first element)."""
    if err is None:
        return None
    if err.dtype != torch.int32 or err.numel() < 1 or not err.is_contiguous():
        raise ValueError("err must be a contiguous int32 tensor of at least one element")
    return err.data_ptr()


def _require_device(*tensors, err=None):
    """Every tensor handed to the library must live on the current CUDA
    device: the library launches there, on that device's stream.  Checked
    last, after the shape checks (the error word's included), so those run on
    any machine."""
    _err_ptr(err)
    tensors = tensors + (err,)
    for v in tensors:
        if v is not None and not v.is_cuda:
            raise ValueError("tensors passed to the library must be CUDA tensors")
    dev = torch.cuda.current_device()
    for v in tensors:
        if v is not None and v.device.index != dev:
            raise ValueError(f"tensors must be on the current CUDA device (cuda:{dev}), "
                             f"got {v.device}")


def slp_forward(x, t, mask=None, T: float = 1.0, logprob=None, lse=None, err=None, stream=None):
    """Forward of the logits-input path.  Returns (logprob[N], lse[N]), float32."""
    N, V, ld = _logits_layout(x)
    _check_vec("t", t, N, torch.int32)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    if logprob is None:
        logprob = torch.empty(N, dtype=torch.float32, device=x.device)
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=x.device)
    _check_vec("logprob", logprob, N, torch.float32)
    _check_vec("lse", lse, N, torch.float32)
    _require_device(x, t, mask, logprob, lse, err=err)
    _lib.call("slp_forward", _ptr(x), _DTYPES[x.dtype], N, V, ld, _ptr(t), _ptr(mask), float(T),
              _ptr(logprob), _ptr(lse), _err_ptr(err), _stream_handle(stream))
    return logprob, lse


def slp_backward(x, t, mask, T: float, lse, grad_out, grad_x=None, err=None, stream=None):
    """Backward of the logits-input path.  Returns grad_x [N, V] (x's dtype)."""
    N, V, ld = _logits_layout(x)
    _check_vec("t", t, N, torch.int32)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    _check_vec("lse", lse, N, torch.float32)
    _check_vec("grad_out", grad_out, N, torch.float32)
    if grad_x is None:
        grad_x = torch.empty((N, V), dtype=x.dtype, device=x.device)
    ldg = _check_grad_x(grad_x, x, N, V)
    _require_device(x, t, mask, lse, grad_out, grad_x, err=err)
    _lib.call("slp_backward", _ptr(x), _DTYPES[x.dtype], N, V, ld, _ptr(t), _ptr(mask), float(T),
              _ptr(lse), _ptr(grad_out), _ptr(grad_x), ldg, _err_ptr(err), _stream_handle(stream))
    return grad_x


def slp_forward_entropy(x, t, mask=None, T: float = 1.0, logprob=None, lse=None, entropy=None,
                        err=None, stream=None):
    """Forward plus per-token entropy.  Returns (logprob, lse, entropy)."""
    N, V, ld = _logits_layout(x)
    _check_vec("t", t, N, torch.int32)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    out = []
    for v in (logprob, lse, entropy):
        v = torch.empty(N, dtype=torch.float32, device=x.device) if v is None else v
        _check_vec("output", v, N, torch.float32)
        out.append(v)
    _require_device(x, t, mask, *out, err=err)
    _lib.call("slp_forward_entropy", _ptr(x), _DTYPES[x.dtype], N, V, ld, _ptr(t), _ptr(mask),
              float(T), _ptr(out[0]), _ptr(out[1]), _ptr(out[2]), _err_ptr(err), _stream_handle(stream))
    return tuple(out)


def slp_backward_entropy(x, t, mask, T: float, lse, entropy, grad_out=None, grad_entropy=None,
                         grad_x=None, err=None, stream=None):
    """Gradient of sum(g * logprob + gH * entropy) with respect to x."""
    N, V, ld = _logits_layout(x)
    _check_vec("t", t, N, torch.int32)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    _check_vec("lse", lse, N, torch.float32)
    _check_vec("entropy", entropy, N, torch.float32)
    for name, v in (("grad_out", grad_out), ("grad_entropy", grad_entropy)):
        if v is not None:
            _check_vec(name, v, N, torch.float32)
    if grad_x is None:
        grad_x = torch.empty((N, V), dtype=x.dtype, device=x.device)
    ldg = _check_grad_x(grad_x, x, N, V)
    _require_device(x, t, mask, lse, entropy, grad_out, grad_entropy, grad_x, err=err)
    _lib.call("slp_backward_entropy", _ptr(x), _DTYPES[x.dtype], N, V, ld, _ptr(t), _ptr(mask),
              float(T), _ptr(lse), _ptr(entropy), _ptr(grad_out), _ptr(grad_entropy),
              _ptr(grad_x), ldg, _err_ptr(err), _stream_handle(stream))
    return grad_x


class _SelectedLogprobEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, t, mask, T):
        lp, lse, H = slp_forward_entropy(x, t, mask, T)
        ctx.save_for_backward(x, t, mask, lse, H)
        ctx.T = T
        ctx.mark_non_differentiable(lse)
        return lp, H, lse

    @staticmethod
    def backward(ctx, g, gH, _g_lse):
        x, t, mask, lse, H = ctx.saved_tensors
        gx = slp_backward_entropy(x, t, mask, ctx.T, lse, H,
                                  None if g is None else g.float().contiguous(),
                                  None if gH is None else gH.float().contiguous())
        return gx, None, None, None


def selected_logprob_and_entropy(x, t, mask=None, temperature: float = 1.0):
    """(logprob[N], entropy[N]) of softmax(x / T) from one read of x, with an
    autograd backward covering both outputs."""
    lp, H, _ = _SelectedLogprobEntropy.apply(x, t, mask, float(temperature))
    return lp, H


def _check_topk(ids, lt, N):
    if ids.dim() != 2 or ids.shape[0] != N or ids.dtype != torch.int32 or not ids.is_contiguous():
        raise ValueError("ids must be a contiguous [N, K] int32 tensor")
    if lt.shape != ids.shape or lt.dtype != torch.float32 or not lt.is_contiguous():
        raise ValueError("teacher_logp must be a contiguous [N, K] float32 tensor")
    return ids.shape[1]


def slp_topk_kl_forward(x, ids, teacher_logp, mask=None, T: float = 1.0,
                        clamp_min: float = float("-inf"), err=None, stream=None):
    """Top-k forward KL.  Returns (kl, student_mass, teacher_mass, lse)."""
    N, V, ld = _logits_layout(x)
    K = _check_topk(ids, teacher_logp, N)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    out = [torch.empty(N, dtype=torch.float32, device=x.device) for _ in range(4)]
    _require_device(x, ids, teacher_logp, mask, *out, err=err)
    _lib.call("slp_topk_kl_forward", _ptr(x), _DTYPES[x.dtype], N, V, ld, _ptr(ids),
              _ptr(teacher_logp), K, _ptr(mask), float(T), float(clamp_min), _ptr(out[0]),
              _ptr(out[1]), _ptr(out[2]), _ptr(out[3]), _err_ptr(err), _stream_handle(stream))
    return tuple(out)


def slp_topk_kl_backward(x, ids, teacher_logp, mask, T: float, clamp_min: float, lse, grad_kl,
                         grad_x=None, err=None, stream=None):
    """Gradient of sum(grad_kl * kl) with respect to x."""
    N, V, ld = _logits_layout(x)
    K = _check_topk(ids, teacher_logp, N)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    _check_vec("lse", lse, N, torch.float32)
    _check_vec("grad_kl", grad_kl, N, torch.float32)
    if grad_x is None:
        grad_x = torch.empty((N, V), dtype=x.dtype, device=x.device)
    ldg = _check_grad_x(grad_x, x, N, V)
    _require_device(x, ids, teacher_logp, mask, lse, grad_kl, grad_x, err=err)
    _lib.call("slp_topk_kl_backward", _ptr(x), _DTYPES[x.dtype], N, V, ld, _ptr(ids),
              _ptr(teacher_logp), K, _ptr(mask), float(T), float(clamp_min), _ptr(lse),
              _ptr(grad_kl), _ptr(grad_x), ldg, _err_ptr(err), _stream_handle(stream))
    return grad_x


def slp_forward_backward(x, t, mask, T: float, grad_out, logprob=None, lse=None, grad_x=None,
                         err=None, stream=None):
    """Forward and backward of the logits-input path in one pass, for an
    upstream gradient known at forward time.  Returns (logprob, lse, grad_x)."""
    N, V, ld = _logits_layout(x)
    _check_vec("t", t, N, torch.int32)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    _check_vec("grad_out", grad_out, N, torch.float32)
    if logprob is None:
        logprob = torch.empty(N, dtype=torch.float32, device=x.device)
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=x.device)
    _check_vec("logprob", logprob, N, torch.float32)
    _check_vec("lse", lse, N, torch.float32)
    if grad_x is None:
        grad_x = torch.empty((N, V), dtype=x.dtype, device=x.device)
    ldg = _check_grad_x(grad_x, x, N, V)
    _require_device(x, t, mask, grad_out, logprob, lse, grad_x, err=err)
    _lib.call("slp_forward_backward", _ptr(x), _DTYPES[x.dtype], N, V, ld, _ptr(t), _ptr(mask),
              float(T), _ptr(grad_out), _ptr(logprob), _ptr(lse), _ptr(grad_x), ldg, _err_ptr(err),
              _stream_handle(stream))
    return logprob, lse, grad_x


def slp_forward_backward_entropy(x, t, mask, T: float, grad_out=None, grad_entropy=None,
                                 logprob=None, lse=None, entropy=None, grad_x=None, err=None,
                                 stream=None):
    """Forward with the entropy and the gradient of sum(g * logprob + gH *
    entropy) in one pass, for weights known at forward time (either may be
    None, meaning zero).  Returns (logprob, lse, entropy, grad_x)."""
    N, V, ld = _logits_layout(x)
    _check_vec("t", t, N, torch.int32)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    for name, v in (("grad_out", grad_out), ("grad_entropy", grad_entropy)):
        if v is not None:
            _check_vec(name, v, N, torch.float32)
    out = []
    for v in (logprob, lse, entropy):
        v = torch.empty(N, dtype=torch.float32, device=x.device) if v is None else v
        _check_vec("output", v, N, torch.float32)
        out.append(v)
    if grad_x is None:
        grad_x = torch.empty((N, V), dtype=x.dtype, device=x.device)
    ldg = _check_grad_x(grad_x, x, N, V)
    _require_device(x, t, mask, grad_out, grad_entropy, *out, grad_x, err=err)
    _lib.call("slp_forward_backward_entropy", _ptr(x), _DTYPES[x.dtype], N, V, ld, _ptr(t),
              _ptr(mask), float(T), _ptr(grad_out), _ptr(grad_entropy), _ptr(out[0]),
              _ptr(out[1]), _ptr(out[2]), _ptr(grad_x), ldg, _err_ptr(err), _stream_handle(stream))
    return out[0], out[1], out[2], grad_x


def slp_lmhead_workspace_size(N: int, V: int, d: int) -> int:
    """Bytes of workspace slp_lmhead_backward needs (enough for the forward too)."""
    return int(_lib.load().slp_lmhead_workspace_size(int(N), int(V), int(d)))


def slp_lmhead_workspace_size_max(N: int, V: int, d: int) -> int:
    """Bytes of workspace with which slp_lmhead_backward runs the whole
    vocabulary as one chunk (fewer launches; the default is 65536 columns)."""
    return int(_lib.load().slp_lmhead_workspace_size_max(int(N), int(V), int(d)))


def slp_lmhead_workspace_size_min(N: int, V: int, d: int) -> int:
    """Least workspace slp_lmhead_backward accepts (vocabulary chunks of 16384
    columns: a quarter of the default dz buffer, for more GEMM launches)."""
    return int(_lib.load().slp_lmhead_workspace_size_min(int(N), int(V), int(d)))


def slp_lmhead_forward_workspace_size(N: int, V: int, d: int) -> int:
    """Bytes of workspace slp_lmhead_forward alone needs."""
    return int(_lib.load().slp_lmhead_forward_workspace_size(int(N), int(V), int(d)))


def slp_lmhead_set_wait_limit_ns(ns: int) -> int:
    """Bound (ns) of every pipeline wait in later LM-head launches; 0 restores
    the two-second default.  Returns the previous bound.  A wait that runs
    out sets SLP_DEVICE_ERR_TIMEOUT in the call's error word."""
    return int(_lib.load().slp_lmhead_set_wait_limit_ns(int(ns)))


def _lmhead_check(h, W):
    if h.dim() != 2 or W.dim() != 2 or h.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise ValueError("h [N, d] and W [V, d] must be bfloat16 matrices")
    if not (h.is_contiguous() and W.is_contiguous()) or h.shape[1] != W.shape[1]:
        raise ValueError("h and W must be contiguous with the same inner size d")
    return h.shape[0], W.shape[0], h.shape[1]


def _workspace(N, V, d, ws, device, forward_only=False):
    """The caller's workspace (any dtype, contiguous) and its size in bytes,
    or a new one of the size the call needs."""
    need = (slp_lmhead_forward_workspace_size if forward_only else slp_lmhead_workspace_size)(N, V, d)
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    if not ws.is_contiguous():
        raise ValueError("ws must be a contiguous tensor")
    return ws, ws.numel() * ws.element_size()


def slp_lmhead_forward(h, W, t, mask=None, T: float = 1.0, logprob=None, lse=None, ws=None,
                       err=None, stream=None):
    """Fused LM-head forward.  Returns (logprob[N], lse[N]), float32."""
    N, V, d = _lmhead_check(h, W)
    _check_vec("t", t, N, torch.int32)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    if logprob is None:
        logprob = torch.empty(N, dtype=torch.float32, device=h.device)
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=h.device)
    _check_vec("logprob", logprob, N, torch.float32)
    _check_vec("lse", lse, N, torch.float32)
    ws, nbytes = _workspace(N, V, d, ws, h.device, forward_only=True)
    _require_device(h, W, t, mask, logprob, lse, ws, err=err)
    _lib.call("slp_lmhead_forward", _ptr(h), _ptr(W), N, V, d, _ptr(t), _ptr(mask), float(T),
              _ptr(logprob), _ptr(lse), _ptr(ws), nbytes, _err_ptr(err), _stream_handle(stream))
    return logprob, lse


def slp_lmhead_forward_noalloc(h, W, t, mask, T: float, logprob, lse, err=None, stream=None):
    """Fused LM-head forward into caller-provided outputs, using the library's
    fixed 16 MiB device scratch instead of a workspace (for callers that cannot
    allocate).  Calls that overlap on the GPU race on that scratch."""
    N, V, d = _lmhead_check(h, W)
    _check_vec("t", t, N, torch.int32)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    _check_vec("logprob", logprob, N, torch.float32)
    _check_vec("lse", lse, N, torch.float32)
    _require_device(h, W, t, mask, logprob, lse, err=err)
    _lib.call("slp_lmhead_forward_noalloc", _ptr(h), _ptr(W), N, V, d, _ptr(t), _ptr(mask),
              float(T), _ptr(logprob), _ptr(lse), _err_ptr(err), _stream_handle(stream))
    return logprob, lse


def slp_lmhead_backward(h, W, t, mask, T: float, lse, grad_out, dh=None, dW=None, ws=None,
                        err=None, stream=None):
    """Fused LM-head backward.  Returns (dh [N, d], dW [V, d]), bfloat16."""
    N, V, d = _lmhead_check(h, W)
    _check_vec("t", t, N, torch.int32)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    _check_vec("lse", lse, N, torch.float32)
    _check_vec("grad_out", grad_out, N, torch.float32)
    if dh is None:
        dh = torch.empty((N, d), dtype=torch.bfloat16, device=h.device)
    if dW is None:
        dW = torch.empty((V, d), dtype=torch.bfloat16, device=h.device)
    _check_mat("dh", dh, N, d, torch.bfloat16)
    _check_mat("dW", dW, V, d, torch.bfloat16)
    _check_disjoint("dh", dh, h, W, dW)
    _check_disjoint("dW", dW, h, W)
    ws, nbytes = _workspace(N, V, d, ws, h.device)
    _require_device(h, W, t, mask, lse, grad_out, dh, dW, ws, err=err)
    _lib.call("slp_lmhead_backward", _ptr(h), _ptr(W), N, V, d, _ptr(t), _ptr(mask), float(T),
              _ptr(lse), _ptr(grad_out), _ptr(dh), _ptr(dW), _ptr(ws), nbytes, _err_ptr(err),
              _stream_handle(stream))
    return dh, dW


def slp_lmhead_backward_accumulate(h, W, t, mask, T: float, lse, grad_out, dW_accum, dh=None,
                                   ws=None, err=None, stream=None):
    """Fused LM-head backward that writes dh and ADDS this micro-batch's dW into
    the float32 accumulator dW_accum [V, d].  Returns dh."""
    N, V, d = _lmhead_check(h, W)
    _check_vec("t", t, N, torch.int32)
    if mask is not None:
        _check_vec("mask", mask, N, torch.uint8)
    _check_vec("lse", lse, N, torch.float32)
    _check_vec("grad_out", grad_out, N, torch.float32)
    _check_mat("dW_accum", dW_accum, V, d, torch.float32)
    if dh is None:
        dh = torch.empty((N, d), dtype=torch.bfloat16, device=h.device)
    _check_mat("dh", dh, N, d, torch.bfloat16)
    _check_disjoint("dh", dh, h, W, dW_accum)
    _check_disjoint("dW_accum", dW_accum, h, W)
    ws, nbytes = _workspace(N, V, d, ws, h.device)
    _require_device(h, W, t, mask, lse, grad_out, dh, dW_accum, ws, err=err)
    _lib.call("slp_lmhead_backward_accumulate", _ptr(h), _ptr(W), N, V, d, _ptr(t), _ptr(mask),
              float(T), _ptr(lse), _ptr(grad_out), _ptr(dh), _ptr(dW_accum), _ptr(ws), nbytes,
              _err_ptr(err), _stream_handle(stream))
    return dh


class _SelectedLogprob(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, t, mask, T):
        lp, lse = slp_forward(x, t, mask, T)
        ctx.save_for_backward(x, t, mask, lse)
        ctx.T = T
        ctx.mark_non_differentiable(lse)
        return lp, lse

    @staticmethod
    def backward(ctx, g, _g_lse):
        x, t, mask, lse = ctx.saved_tensors
        gx = slp_backward(x, t, mask, ctx.T, lse, g.float().contiguous())
        return gx, None, None, None


def selected_logprob(x, t, mask=None, temperature: float = 1.0):
    """logprob[N] = log_softmax(x / T)[n, t_n] with an autograd backward that
    recomputes the softmax from x and the saved lse (no [N, V] float buffer).
    Rows with mask == 0 give 0 and a zero gradient."""
    lp, _ = _SelectedLogprob.apply(x, t, mask, float(temperature))
    return lp


class _LMHeadSelectedLogprob(torch.autograd.Function):
    @staticmethod
    def forward(ctx, h, W, t, mask, T):
        lp, lse = slp_lmhead_forward(h, W, t, mask, T)
        ctx.save_for_backward(h, W, t, mask, lse)
        ctx.T = T
        ctx.mark_non_differentiable(lse)
        return lp, lse

    @staticmethod
    def backward(ctx, g, _g_lse):
        h, W, t, mask, lse = ctx.saved_tensors
        dh, dW = slp_lmhead_backward(h, W, t, mask, ctx.T, lse, g.float().contiguous())
        return dh, dW, None, None, None


def lmhead_selected_logprob(h, W, t, mask=None, temperature: float = 1.0):
    """Selected-token log-probabilities of the logits h W^T / T without storing
    them; only rows with mask != 0 are projected."""
    lp, _ = _LMHeadSelectedLogprob.apply(h, W, t, mask, float(temperature))
    return lp
