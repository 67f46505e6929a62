"""GPU: slp_lmhead_forward_noalloc, the LM-head forward for callers that cannot
allocate device memory (their framework owns all of it, or cudaMalloc's
device-wide synchronisation is not acceptable where they call from).  It must
give the same results as slp_lmhead_forward with a caller workspace, on two
calls in a row that share the library's fixed scratch.

Kept in its own file, collected last, so a failure here leaves every other
test already run."""

import ctypes

import numpy as np
import pytest
import torch

import vocab_selected_token_gb300 as slp
from tests.gpu_util import device
from vocab_selected_token_gb300 import _lib
from vocab_selected_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_LP = 5e-3  # the LM-head path's logprob tolerance


def _noalloc(lib, a, lp, lse, err):
    N, d = a.h.shape
    V = a.W.shape[0]
    return lib.slp_lmhead_forward_noalloc(
        a.h.data_ptr(), a.W.data_ptr(), N, V, d, a.t.data_ptr(), a.mask.data_ptr(),
        float(a.T), lp.data_ptr(), lse.data_ptr(), err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_forward_on_two_calls():
    dev = device()
    lib = _lib.load()
    cases = [W.make_lmhead_inputs(device=dev, N=700, V=9000, d=256, seed=21),
             W.make_lmhead_inputs(device=dev, N=1000, V=151936, d=2560, seed=22, p_mask=0.7)]
    for a in cases:
        N = a.h.shape[0]
        lp = torch.full((N,), 9.0, device=dev)
        lse = torch.full((N,), 9.0, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        assert _noalloc(lib, a, lp, lse, err) == _lib.SLP_OK
        ref_lp, ref_lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert bool(torch.isfinite(lp).all()) and bool(torch.isfinite(lse).all())
        assert float((lp - ref_lp).abs().max()) <= TOL_LP
        assert float((lse - ref_lse).abs().max()) <= TOL_LP
        off = a.mask == 0
        assert bool((lp[off] == 0).all()) and bool((lse[off] == 0).all())


def test_noalloc_rejects_sizes_beyond_its_scratch():
    device()
    lib = _lib.load()
    N, V, d = 4096, 151936, 2560
    assert slp.slp_lmhead_forward_workspace_size(N, V, d) > (16 << 20)
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: rejected before any launch
    st = lib.slp_lmhead_forward_noalloc(fake, fake, N, V, d, fake, None, 1.0, fake, fake, None,
                                        None)
    assert st == _lib.SLP_ERR_WORKSPACE
