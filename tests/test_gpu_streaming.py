"""GPU: forward_backward_from_host / slp_forward_backward_host (row chunks
streamed from pinned host memory on three overlapping streams) gives the
device call's results, bit for bit."""

import numpy as np
import pytest
import torch

import vocab_selected_token_gb300 as slp
from tests.gpu_util import check_rows, device
from vocab_selected_token_gb300 import workloads as W
from vocab_selected_token_gb300.streaming import forward_backward_from_host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,N,V,R", [("c151k", 300, 151936, 64), ("packed", 1000, 20016, 128),
                                        ("stability", 97, 131072, 40), ("tiny", 5, 2047, 2)])
def test_streaming_matches_device_call(name, N, V, R):
    dev = device()
    a = W.make_logits_inputs(name, device=dev, N=N, V=V)
    xh = a.x.cpu().pin_memory()
    th = a.t.cpu().pin_memory()
    gh = a.g.cpu().pin_memory()
    mh = None if a.mask is None else a.mask.cpu().pin_memory()
    lp, lse, gx = forward_backward_from_host(xh, th, gh, mh, a.T, rows_per_chunk=R)
    lp_d, lse_d, gx_d = slp.slp_forward_backward(a.x, a.t, a.mask, a.T, a.g)
    torch.cuda.synchronize()
    assert torch.equal(lp, lp_d.cpu()) and torch.equal(lse, lse_d.cpu())
    assert torch.equal(gx, gx_d.cpu())
    rows = set(np.random.default_rng(3).choice(N, min(N, 12), replace=False).tolist())
    check_rows(a.x, a.t, a.mask, a.T, a.g, lp_d, lse_d, gx_d, rows)


def test_streaming_padded_rows_and_default_chunk():
    """Rows with a stride wider than V on both sides, and the library's own
    chunk size (several chunks at this N)."""
    dev = device()
    N, V, pad = 200, 151936, 24
    a = W.make_logits_inputs("c151k", device=dev, N=N, V=V)
    xh_full = torch.zeros((N, V + pad), dtype=a.x.dtype).pin_memory()
    xh_full[:, :V] = a.x.cpu()
    gx_full = torch.full((N, V + pad), 7.0, dtype=a.x.dtype).pin_memory()
    th, gh = a.t.cpu().pin_memory(), a.g.cpu().pin_memory()
    lp, lse, gx = forward_backward_from_host(xh_full[:, :V], th, gh, None, a.T,
                                             grad_x=gx_full[:, :V])
    lp_d, lse_d, gx_d = slp.slp_forward_backward(a.x, a.t, None, a.T, a.g)
    torch.cuda.synchronize()
    assert torch.equal(lp, lp_d.cpu()) and torch.equal(lse, lse_d.cpu())
    assert torch.equal(gx_full[:, :V], gx_d.cpu())
    assert bool((gx_full[:, V:] == 7.0).all())  # the padding is not written


def test_streaming_rejects_pageable_host_memory():
    """The C entry point refuses host buffers that are not page-locked."""
    from vocab_selected_token_gb300 import _lib
    dev = device()
    N, V = 8, 256
    lib = _lib.load()
    x = torch.zeros((N, V), dtype=torch.bfloat16)  # pageable
    t = torch.zeros(N, dtype=torch.int32).pin_memory()
    g = torch.zeros(N).pin_memory()
    lp, lse = torch.zeros(N).pin_memory(), torch.zeros(N).pin_memory()
    gx = torch.zeros((N, V), dtype=torch.bfloat16).pin_memory()
    ws_b = lib.slp_forward_backward_host_workspace_size(N, V, 0, 0)
    ws = torch.empty(ws_b, dtype=torch.uint8, device=dev)
    st = lib.slp_forward_backward_host(x.data_ptr(), 0, N, V, V, t.data_ptr(), None, 1.0,
                                       g.data_ptr(), lp.data_ptr(), lse.data_ptr(), gx.data_ptr(),
                                       V, 0, ws.data_ptr(), ws_b, None, None)
    assert st == _lib.SLP_ERR_INVALID_ARG
    st = lib.slp_forward_backward_host(x.pin_memory().data_ptr(), 0, N, V, V, t.data_ptr(), None,
                                       1.0, g.data_ptr(), lp.data_ptr(), lse.data_ptr(),
                                       gx.data_ptr(), V, 0, ws.data_ptr(), ws_b - 256, None, None)
    assert st == _lib.SLP_ERR_WORKSPACE
