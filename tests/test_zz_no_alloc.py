"""GPU: slp_lmhead_forward_noalloc, the LM-head forward for callers that cannot
allocate device memory (their framework owns all of it, or cudaMalloc's
device-wide synchronisation is not acceptable where they call from).  It must
give the same results as slp_lmhead_forward with a caller workspace, on two
calls in a row that share the library's fixed scratch, and match the fp64
oracle on calls that run over what earlier calls left in that scratch.

Kept in its own file, collected last, so a failure here leaves every other
test already run."""

import ctypes

import numpy as np
import pytest
import torch

import vocab_selected_token_gb300 as slp
from oracle import slp_oracle as O
from tests.gpu_util import assert_close_nan, device, to64
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


def test_noalloc_against_the_oracle_on_reused_scratch():
    """Three calls in a row on the shared scratch, each checked row by row
    against the fp64 oracle: a case at the scratch's limit (N = 1792 at
    V = 151936, d = 2560, every row active), a smaller one with another mask
    density and temperature that runs on the first call's leftovers, and the
    first case again on the second's.  Masked rows must be exactly +0.0."""
    dev = device()
    lib = _lib.load()
    N, V, d = 1792, 151936, 2560
    assert slp.slp_lmhead_forward_workspace_size(N, V, d) <= (16 << 20)
    big = W.make_lmhead_inputs(device=dev, N=N, V=V, d=d, seed=31, p_mask=1.0)
    small = W.make_lmhead_inputs(device=dev, N=900, V=V, d=d, seed=32, p_mask=0.3)
    small.T = 0.7
    W64 = to64(big.W)
    refs = {}
    for name, a in (("big", big), ("small", small), ("big again", big)):
        n = a.h.shape[0]
        lp = torch.full((n,), 9.0, device=dev)
        lse = torch.full((n,), 9.0, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        assert _noalloc(lib, a, lp, lse, err) == _lib.SLP_OK
        torch.cuda.synchronize()
        assert int(err.item()) == 0, name
        key = "small" if a is small else "big"
        if key not in refs:
            Wa = W64 if a is big else to64(a.W)
            refs[key] = O.lmhead_forward(to64(a.h), Wa, a.t.cpu().numpy(), a.mask.cpu().numpy(),
                                         a.T)
        rlp, rlse = refs[key]
        assert_close_nan(to64(lp), rlp, TOL_LP, f"logprob ({name})")
        assert_close_nan(to64(lse), rlse, TOL_LP, f"lse ({name})")
        off = a.mask == 0
        assert bool((lp[off].view(torch.int32) == 0).all()), f"masked logprob not +0.0 ({name})"
        assert bool((lse[off].view(torch.int32) == 0).all()), f"masked lse not +0.0 ({name})"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    device()
    lib = _lib.load()
    N, V, d = 4096, 151936, 2560
    assert slp.slp_lmhead_forward_workspace_size(N, V, d) > (16 << 20)
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: rejected before any launch
    st = lib.slp_lmhead_forward_noalloc(fake, fake, N, V, d, fake, None, 1.0, fake, fake, None,
                                        None)
    assert st == _lib.SLP_ERR_WORKSPACE
