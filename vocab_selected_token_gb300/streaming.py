"""Selected-token log-probabilities for logits that live in host memory.

When the logits of a large micro-batch sit in (pinned) host memory, for
example after a CPU offload, `forward_backward_from_host` streams them through
the GPU in row chunks.  Three CUDA streams run at once:

    copy-in   : chunk k's logits, targets, mask and upstream gradient -> device
    compute   : slp_forward_backward on chunk k-1 (one read of the logits)
    copy-out  : chunk k-2's logprob, lse and gradient -> host

so the two directions of the host link and the kernels overlap.  Device
buffers for `slots` chunks are allocated once per call and reused round-robin;
events order every reuse.  All arithmetic runs in the library's CUDA kernels;
this module only moves bytes and orders streams.
"""

from __future__ import annotations

import torch

from . import slp_forward_backward


def forward_backward_from_host(x, t, grad_out, mask=None, T: float = 1.0, *,
                               logprob=None, lse=None, grad_x=None,
                               rows_per_chunk: int | None = None, slots: int = 3,
                               device=None):
    """Forward and backward of the selected-token log-probability for host
    tensors.

    x [N, V] (bf16 or f32), t [N] int32, grad_out [N] f32 and mask [N] uint8
    (optional) must be pinned CPU tensors.  Results go to pinned host tensors
    (allocated when not given): logprob [N], lse [N] f32 and grad_x [N, V] in
    x's dtype.  Returns (logprob, lse, grad_x); they are complete when this
    function returns (it synchronises on its own streams at the end).
    """
    if device is None:
        device = torch.device("cuda", torch.cuda.current_device())
    for name, v in (("x", x), ("t", t), ("grad_out", grad_out), ("mask", mask)):
        if v is not None and (v.is_cuda or not v.is_pinned()):
            raise ValueError(f"{name} must be a pinned host tensor")
    N, V = x.shape
    if logprob is None:
        logprob = torch.empty(N, dtype=torch.float32).pin_memory()
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32).pin_memory()
    if grad_x is None:
        grad_x = torch.empty((N, V), dtype=x.dtype).pin_memory()
    if N == 0:
        return logprob, lse, grad_x
    if rows_per_chunk is None:
        # about 64 MB of logits per chunk: short pipeline fill and drain
        rows_per_chunk = max(1, (64 << 20) // max(1, V * x.element_size()))
    R = min(rows_per_chunk, N)
    nchunks = (N + R - 1) // R
    slots = max(1, min(slots, nchunks))

    s_in = torch.cuda.Stream(device)
    s_cmp = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    bufs = []
    for _ in range(slots):
        bufs.append({
            "x": torch.empty((R, V), dtype=x.dtype, device=device),
            "t": torch.empty(R, dtype=torch.int32, device=device),
            "g": torch.empty(R, dtype=torch.float32, device=device),
            "m": None if mask is None else torch.empty(R, dtype=torch.uint8, device=device),
            "lp": torch.empty(R, dtype=torch.float32, device=device),
            "lse": torch.empty(R, dtype=torch.float32, device=device),
            "gx": torch.empty((R, V), dtype=x.dtype, device=device),
            "in_done": torch.cuda.Event(),
            "cmp_done": torch.cuda.Event(),
            "out_done": None,
        })
    for k in range(nchunks):
        b = bufs[k % slots]
        r0, r1 = k * R, min(N, (k + 1) * R)
        n = r1 - r0
        # copy-in may reuse the slot once the chunk that used it is copied out
        with torch.cuda.stream(s_in):
            if b["out_done"] is not None:
                s_in.wait_event(b["out_done"])
            b["x"][:n].copy_(x[r0:r1], non_blocking=True)
            b["t"][:n].copy_(t[r0:r1], non_blocking=True)
            b["g"][:n].copy_(grad_out[r0:r1], non_blocking=True)
            if mask is not None:
                b["m"][:n].copy_(mask[r0:r1], non_blocking=True)
            b["in_done"].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(b["in_done"])
            slp_forward_backward(b["x"][:n], b["t"][:n], None if mask is None else b["m"][:n],
                                 T, b["g"][:n], logprob=b["lp"][:n], lse=b["lse"][:n],
                                 grad_x=b["gx"][:n], stream=s_cmp)
            b["cmp_done"].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(b["cmp_done"])
            logprob[r0:r1].copy_(b["lp"][:n], non_blocking=True)
            lse[r0:r1].copy_(b["lse"][:n], non_blocking=True)
            grad_x[r0:r1].copy_(b["gx"][:n], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s_out)
            b["out_done"] = ev
    s_out.synchronize()
    s_cmp.synchronize()
    s_in.synchronize()
    return logprob, lse, grad_x
