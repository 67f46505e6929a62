"""GPU: the bounds-checked build (libslp_checked.so, -DSLP_DEBUG_BOUNDS).

In that build every kernel checks each global load and store against the
byte ranges of the buffers its call was given, skips an access outside all
of them and reports it with SLP_DEVICE_ERR_BOUNDS in the error word; nothing
traps.  It stands in for a memory checker.  These tests run the tiny workload,
the scaled recipes (many tiles, ragged vocabulary tails, unaligned rows,
short rows, cluster-split rows), the fused, entropy and top-k calls and small
LM-head cases through the checked library's C ABI (the Python binding pointed
at it), and require a clean error word and oracle parity at the usual
tolerances.  A self-test shows that the checks do refuse an access outside
the permitted ranges."""

from __future__ import annotations

import contextlib
import ctypes

import numpy as np
import pytest
import torch

import vocab_selected_token_gb300 as slp
from oracle import slp_oracle as O
from tests.gpu_util import assert_close_nan, assert_grad_close, check_rows, device, to64
from tests import test_gpu_lmhead_random as LMR
from tests.test_gpu_entropy import check_entropy_rows
from tests.test_gpu_random_shapes import run_shape
from vocab_selected_token_gb300 import _lib, build
from vocab_selected_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@contextlib.contextmanager
def checked_library():
    """Route the binding's calls to libslp_checked.so for the duration."""
    device()
    path = build.build_checked()
    lib = ctypes.CDLL(path)
    for name, (res, args) in _lib.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    saved = _lib.load()
    _lib._lib = lib
    try:
        yield lib
    finally:
        torch.cuda.synchronize()
        _lib._lib = saved


def clean(err):
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & _lib.SLP_DEVICE_ERR_BOUNDS == 0, "an access outside the call's buffers"
    assert e == 0, f"error word {e}"


def test_checked_build_refuses_an_access_outside_the_table():
    dev = device()
    buf = torch.full((8,), 5.0, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = _lib.load().slp_bounds_check_selftest(buf.data_ptr(), err.data_ptr(), None)
    assert st == _lib.SLP_ERR_UNSUPPORTED  # the normal build has no checks
    with checked_library() as lib:
        assert lib.slp_bounds_check_selftest(buf.data_ptr(), err.data_ptr(), None) == _lib.SLP_OK
        torch.cuda.synchronize()
    assert int(err.item()) == _lib.SLP_DEVICE_ERR_BOUNDS
    assert float(buf[4]) == 5.0 and float(buf[0]) == 1.0


LOGITS = [
    ("tiny", None, None),
    ("c151k", 48, 151936),         # cluster-split rows
    ("c151k", 33, 151936 - 5),     # ragged vector tail
    ("packed", 3000, 20016),       # masked spans, warp-per-row kernels
    ("stability", 256, 131072),    # fp32, -inf columns; fused: TMEM part, 4 CTAs
    ("stability", 20, 100000),     # fp32, fused: TMEM part, 3 CTAs per row instead of 6
    ("tiny", 4, 560000),           # 1.09 MB bf16 rows: the fused call's TMEM form, 8 CTAs
    ("stability", 64, 4099),
    ("tiny", 300, 2047),           # rows not 16-byte aligned: scalar kernels
]


@pytest.mark.parametrize("name,N,V", LOGITS, ids=lambda v: str(v))
def test_logits_calls_stay_in_bounds(name, N, V):
    dev = device()
    a = W.make_logits_inputs(name, device=dev, N=N, V=V)
    n = a.x.shape[0]
    with checked_library():
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        lp, lse = slp.slp_forward(a.x, a.t, a.mask, a.T, err=err)
        gx = slp.slp_backward(a.x, a.t, a.mask, a.T, lse, a.g, err=err)
        clean(err)
        check_rows(a.x, a.t, a.mask, a.T, a.g, lp, lse, gx, range(n))
        lp2, lse2, gx2 = slp.slp_forward_backward(a.x, a.t, a.mask, a.T, a.g, err=err)
        clean(err)
        check_rows(a.x, a.t, a.mask, a.T, a.g, lp2, lse2, gx2, range(n))
        gH = torch.linspace(-1.0, 1.0, n, device=dev)
        lp3, lse3, H3 = slp.slp_forward_entropy(a.x, a.t, a.mask, a.T, err=err)
        gx3 = slp.slp_backward_entropy(a.x, a.t, a.mask, a.T, lse3, H3, a.g, gH, err=err)
        _, _, H4, gx4 = slp.slp_forward_backward_entropy(a.x, a.t, a.mask, a.T, a.g, gH,
                                                          err=err)
        clean(err)
    check_entropy_rows(a, gH, lp3, lse3, H3, gx3, range(n))
    check_entropy_rows(a, gH, lp3, lse3, H4, gx4, range(n))


def test_short_rows_and_topk_stay_in_bounds():
    dev = device()
    a = W.make_logits_inputs("tiny", device=dev, N=600, V=4096)  # warp-per-row kernels
    k = W.make_topk_inputs(device=dev, N=96, V=2048, K=32)
    with checked_library():
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        lp, lse, gx = slp.slp_forward_backward(a.x, a.t, None, a.T, a.g, err=err)
        clean(err)
        check_rows(a.x, a.t, None, a.T, a.g, lp, lse, gx, range(600))
        kl, sm, tm, klse = slp.slp_topk_kl_forward(k.x, k.ids, k.lt, None, k.T, k.clamp,
                                                   err=err)
        gk = slp.slp_topk_kl_backward(k.x, k.ids, k.lt, None, k.T, k.clamp, klse, k.g, err=err)
        clean(err)
    x64 = to64(k.x)
    ids = k.ids.cpu().numpy()
    lt = to64(k.lt)
    rkl, rsm, rtm, rlse = O.topk_kl_forward(x64, ids, lt, None, k.T, k.clamp)
    assert_close_nan(to64(kl), rkl, 5e-5, "kl")
    assert_close_nan(to64(sm), rsm, 5e-5, "student mass")
    rgk = O.topk_kl_backward(x64, ids, lt, None, k.T, k.clamp, rlse, to64(k.g))
    assert_grad_close(to64(gk), rgk, "top-k gradient")


@pytest.mark.parametrize("N,V,d,pm", [(300, 1000, 128, 0.5), (130, 4096, 2560, 0.9)],
                         ids=lambda v: str(v))
def test_lmhead_calls_stay_in_bounds(N, V, d, pm):
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=N, V=V, d=d, p_mask=pm, seed=13)
    with checked_library():
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        lp, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T, err=err)
        dh, dW = slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, lse, a.g, err=err)
        acc = torch.zeros((V, d), device=dev)
        dh2 = slp.slp_lmhead_backward_accumulate(a.h, a.W, a.t, a.mask, a.T, lse, a.g, acc,
                                                 err=err)
        lp_n = torch.empty(N, device=dev)
        lse_n = torch.empty(N, device=dev)
        slp.slp_lmhead_forward_noalloc(a.h, a.W, a.t, a.mask, a.T, lp_n, lse_n, err=err)
        clean(err)
    h64, W64 = to64(a.h), to64(a.W)
    t, m, g = a.t.cpu().numpy(), a.mask.cpu().numpy(), to64(a.g)
    rlp, rlse = O.lmhead_forward(h64, W64, t, m, a.T)
    for got, what in ((lp, "logprob"), (lp_n, "logprob (no-allocation call)")):
        assert_close_nan(to64(got), rlp, 5e-3, what)
    rdh, rdW = O.lmhead_backward(h64, W64, t, m, a.T, rlse, g)
    for got, ref, what in ((dh, rdh, "dh"), (dW, rdW, "dW"), (dh2, rdh, "dh (accumulate)"),
                           (acc, rdW, "dW accumulated")):
        got = to64(got).ravel()
        ref = ref.ravel()
        cos = float(got @ ref / (np.linalg.norm(got) * np.linalg.norm(ref)))
        frob = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
        assert cos >= 0.999 and frob <= 1e-2, f"{what}: cosine {cos:.6f} frob {frob:.2e}"


@pytest.mark.parametrize("seed", range(24))
def test_random_logits_shapes_stay_in_bounds(seed):
    """The seeded sweep of random shapes, strides, dtypes, temperatures and
    mask densities (V from 1 to 160000, padded rows) through the checked
    library: clean error words and oracle parity."""
    dev = device()
    with checked_library():
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        run_shape(seed, err=err)
        clean(err)


@pytest.mark.parametrize("case", [LMR._case(s) for s in range(16)] + LMR.EDGES,
                         ids=lambda v: str(v))
def test_random_lmhead_shapes_stay_in_bounds(case):
    """The LM head's random sweep and edge cases (ragged row blocks, V = 1,
    d not a multiple of the tile, several backward chunks) through the
    checked library."""
    dev = device()
    with checked_library():
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        LMR._run(*case, seed=500 + sum(int(v) for v in case[:3]), err=err)
        clean(err)
