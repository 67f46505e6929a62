"""GPU: forward_backward_from_host (row chunks streamed from pinned host
memory on three overlapping streams) gives the device call's results."""

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
