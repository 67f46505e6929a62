"""Selected-token log-probabilities for logits that live in host memory.

When the logits of a large micro-batch sit in pinned host memory, for
example after a CPU offload, `forward_backward_from_host` streams them through
the GPU in row chunks with the library's `slp_forward_backward_host`.  Three
CUDA streams overlap:

    copy-in   : chunk k+1's logits, targets, mask and upstream gradient -> device
    compute   : slp_forward_backward on chunk k (one read of the logits)
    copy-out  : chunk k-1's logprob, lse and gradient -> host

so both directions of the host link and the kernels run at once.  The
pipeline (chunking, copies, events) is native code.  This module only
allocates the device workspace and the pinned results, and marshals
arguments.
"""

from __future__ import annotations

import torch

from . import _DTYPES, _lib, _ptr


def forward_backward_from_host(x, t, grad_out, mask=None, T: float = 1.0, *,
                               logprob=None, lse=None, grad_x=None,
                               rows_per_chunk: int | None = None, device=None, stream=None):
    """Forward and backward of the selected-token log-probability for host
    tensors.

    x [N, V] (bf16 or f32, unit column stride), t [N] int32, grad_out [N] f32
    and mask [N] uint8 (optional) must be pinned CPU tensors.  Results go to
    pinned host tensors, allocated when not given: logprob [N], lse [N] f32 and
    grad_x [N, V] in x's dtype.  rows_per_chunk=None lets the library pick
    about 64 MB of logits per chunk.  Returns (logprob, lse, grad_x), complete
    when this function returns: it synchronises the stream it used.
    """
    if device is None:
        device = torch.device("cuda", torch.cuda.current_device())
    for name, v in (("x", x), ("t", t), ("grad_out", grad_out), ("mask", mask)):
        if v is not None and (v.is_cuda or not v.is_pinned()):
            raise ValueError(f"{name} must be a pinned host tensor")
    if x.dim() != 2 or x.dtype not in _DTYPES:
        raise ValueError("x must be a 2-D bfloat16 or float32 tensor")
    N, V = x.shape
    if N > 0 and V > 0 and x.stride(1) != 1:
        raise ValueError("x must have unit column stride")
    ld = x.stride(0) if N > 1 else max(V, 1)
    for name, v, dt in (("t", t, torch.int32), ("grad_out", grad_out, torch.float32),
                        ("mask", mask, torch.uint8)):
        if v is not None and (v.shape != (N,) or v.dtype != dt or not v.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous [{N}] {dt} tensor")
    if logprob is None:
        logprob = torch.empty(N, dtype=torch.float32).pin_memory()
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32).pin_memory()
    if grad_x is None:
        grad_x = torch.empty((N, V), dtype=x.dtype).pin_memory()
    if grad_x.shape != (N, V) or grad_x.dtype != x.dtype or (N > 0 and V > 0 and grad_x.stride(1) != 1):
        raise ValueError("grad_x must be [N, V] with x's dtype and unit column stride")
    ldg = grad_x.stride(0) if N > 1 else max(V, 1)
    if N == 0:
        return logprob, lse, grad_x
    dt = _DTYPES[x.dtype]
    rpc = 0 if rows_per_chunk is None else int(rows_per_chunk)
    lib = _lib.load()
    ws_bytes = int(lib.slp_forward_backward_host_workspace_size(N, V, dt, rpc))
    with torch.cuda.device(device):
        s = torch.cuda.current_stream(device) if stream is None else stream
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        _lib.call("slp_forward_backward_host", _ptr(x), dt, N, V, ld, _ptr(t), _ptr(mask),
                  float(T), _ptr(grad_out), _ptr(logprob), _ptr(lse), _ptr(grad_x), ldg, rpc,
                  _ptr(ws), ws_bytes, None, s.cuda_stream)
        s.synchronize()
    return logprob, lse, grad_x
