"""GPU: the calls contain no allocation or host synchronisation, so they can be
captured in a CUDA graph; replaying the graph gives the eager results."""

import pytest
import torch

import vocab_selected_token_gb300 as slp
from tests.gpu_util import device
from vocab_selected_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_logits_path_in_a_cuda_graph():
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev, N=256)
    lp = torch.empty(256, device=dev)
    lse = torch.empty(256, device=dev)
    gx = torch.empty_like(a.x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # warm up outside the capture
        slp.slp_forward(a.x, a.t, None, a.T, logprob=lp, lse=lse, stream=s)
        slp.slp_backward(a.x, a.t, None, a.T, lse, a.g, grad_x=gx, stream=s)
    s.synchronize()
    ref = (lp.clone(), lse.clone(), gx.clone())
    lp.zero_(); lse.zero_(); gx.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        slp.slp_forward(a.x, a.t, None, a.T, logprob=lp, lse=lse, stream=s)
        slp.slp_backward(a.x, a.t, None, a.T, lse, a.g, grad_x=gx, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(lp, ref[0]) and torch.equal(lse, ref[1]) and torch.equal(gx, ref[2])


def test_lmhead_forward_in_a_cuda_graph():
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=300, V=4000, d=256)
    ws = torch.empty(slp.slp_lmhead_workspace_size(300, 4000, 256), dtype=torch.uint8, device=dev)
    lp = torch.empty(300, device=dev)
    lse = torch.empty(300, device=dev)
    dh = torch.empty_like(a.h)
    dW = torch.empty_like(a.W)
    s = torch.cuda.Stream()
    def run():
        slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T, logprob=lp, lse=lse, ws=ws, stream=s)
        slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, lse, a.g, dh=dh, dW=dW, ws=ws, stream=s)
    with torch.cuda.stream(s):
        run()
    s.synchronize()
    ref = [v.clone() for v in (lp, lse, dh, dW)]
    for v in (lp, lse, dh, dW):
        v.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    g.replay()
    torch.cuda.synchronize()
    for v, r in zip((lp, lse, dh, dW), ref):
        assert torch.equal(v, r)
