"""GPU parity of the logits-input path (slp_forward / slp_backward through the
C ABI) against the CPU oracle."""

from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import vocab_selected_token_gb300 as slp
from oracle import slp_oracle as O
from tests.gpu_util import (TOL_LP, assert_close_nan, assert_grad_close, check_rows, device,
                            to64)
from vocab_selected_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "oracle_cases.json")))["cases"]


def run(x, t, mask, T, g, stream=None):
    lp, lse = slp.slp_forward(x, t, mask, T, stream=stream)
    gx = slp.slp_backward(x, t, mask, T, lse, g, stream=stream)
    torch.cuda.synchronize()
    return lp, lse, gx


@pytest.mark.parametrize("case", GOLDEN, ids=lambda c: c["name"])
def test_golden_cases(case):
    dev = device()
    x = torch.tensor(case["x"], dtype=torch.float32, device=dev)
    t = torch.tensor(case["t"], dtype=torch.int32, device=dev)
    g = torch.tensor(case["g"], dtype=torch.float32, device=dev)
    lp, lse, gx = run(x, t, None, case["T"], g)
    assert_close_nan(to64(lp), case["logprob"], TOL_LP, "logprob")
    assert_close_nan(to64(lse), case["lse"], TOL_LP, "lse")
    assert_grad_close(to64(gx), np.array(case["grad_x"]))


def test_tiny_all_rows():
    dev = device()
    a = W.make_logits_inputs("tiny", device=dev)
    lp, lse, gx = run(a.x, a.t, a.mask, a.T, a.g)
    check_rows(a.x, a.t, a.mask, a.T, a.g, lp, lse, gx, range(a.x.shape[0]))


# Same recipes at sizes the oracle handles in seconds, spanning many tiles
# and ragged tails.
SCALED = [
    ("c151k", 48, 151936),
    ("c151k", 33, 151936 - 5),     # V not a multiple of the vector width
    ("packed", 3000, 20016),
    ("stability", 256, 131072),
    ("stability", 64, 4099),
    ("tiny", 300, 2047),           # odd V, rows not 16-byte aligned
]


@pytest.mark.parametrize("name,N,V", SCALED, ids=lambda v: str(v))
def test_scaled_workloads_all_rows(name, N, V):
    dev = device()
    a = W.make_logits_inputs(name, device=dev, N=N, V=V)
    lp, lse, gx = run(a.x, a.t, a.mask, a.T, a.g)
    check_rows(a.x, a.t, a.mask, a.T, a.g, lp, lse, gx, range(N))


def test_ragged_tail_on_vector_path():
    """V not a multiple of 8 but the row stride is: 128-bit body plus scalar
    tail, and the padding columns of grad_x are left untouched."""
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev, N=40, V=20016)
    V = 20011
    x = a.x[:, :V]
    gx = torch.full((40, 20016), 7.0, dtype=torch.bfloat16, device=dev)
    lp, lse = slp.slp_forward(x, a.t % V, None, a.T)
    slp.slp_backward(x, a.t % V, None, a.T, lse, a.g, grad_x=gx[:, :V])
    torch.cuda.synchronize()
    assert bool((gx[:, V:] == 7.0).all()), "columns >= V of grad_x were written"
    check_rows(x, a.t % V, None, a.T, a.g, lp, lse, gx[:, :V], range(40))


# Short rows through the separate kernels: the warp-per-row forward and, where
# the backward's 16 KB tiles would be under 90 % full, the warp-per-row
# backward (including a 40 KB row, masked spans and fp32).
SHORT = [
    ("packed", 70, 200),
    ("tiny", 37, 1000),
    ("c151k", 41, 6144),
    ("c151k", 24, 20480),
    ("stability", 29, 2048),
    ("stability", 20, 5000),
]


@pytest.mark.parametrize("name,N,V", SHORT, ids=lambda v: str(v))
def test_short_rows_all_rows(name, N, V):
    dev = device()
    a = W.make_logits_inputs(name, device=dev, N=N, V=V)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse = slp.slp_forward(a.x, a.t, a.mask, a.T, err=err)
    gx = slp.slp_backward(a.x, a.t, a.mask, a.T, lse, a.g, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_rows(a.x, a.t, a.mask, a.T, a.g, lp, lse, gx, range(N))
    if a.mask is not None:
        assert bool((gx[a.mask == 0].view(torch.int16) == 0).all())


def test_short_rows_ragged_tail_targets_in_tail():
    """8 KB rows with V not a multiple of 8 on a 16-byte-aligned stride, some
    targets among the trailing elements; grad_x's padding left untouched."""
    dev = device()
    V, Vp = 4101, 4104
    a = W.make_logits_inputs("c151k", device=dev, N=48, V=Vp)
    x = a.x[:, :V]
    t = a.t % V
    t[:8] = V - 1 - torch.arange(8, dtype=torch.int32, device=dev) % 5
    gx = torch.full((48, Vp), 7.0, dtype=torch.bfloat16, device=dev)
    lp, lse = slp.slp_forward(x, t, None, a.T)
    slp.slp_backward(x, t, None, a.T, lse, a.g, grad_x=gx[:, :V])
    torch.cuda.synchronize()
    assert bool((gx[:, V:] == 7.0).all())
    check_rows(x, t, None, a.T, a.g, lp, lse, gx[:, :V], range(48))


FULL = ["c151k", "packed", "stability"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(name):
    """Full workload sizes, in the launch configuration the bench times:
    sampled rows against the oracle, every row against properties."""
    dev = device()
    a = W.make_logits_inputs(name, device=dev)
    N, V = a.x.shape
    lp, lse, gx = run(a.x, a.t, a.mask, a.T, a.g)
    gen = np.random.default_rng(17)
    rows = set(gen.choice(N, 40, replace=False).tolist()) | {0, N - 1}
    if name == "stability":
        inf_rows = torch.nonzero(torch.isinf(a.x).any(dim=1))[:, 0].cpu().numpy()
        rows |= set(inf_rows[:8].tolist())
    if a.mask is not None:
        m = a.mask.cpu().numpy()
        edges = np.flatnonzero(np.diff(m.astype(np.int8)))
        rows |= set(edges[:8].tolist()) | set((edges[:8] + 1).tolist())
    check_rows(a.x, a.t, a.mask, a.T, a.g, lp, lse, gx, rows)
    active = torch.ones(N, dtype=torch.bool, device=dev) if a.mask is None else a.mask != 0
    assert bool(torch.isfinite(lp[active]).all()) and bool((lp[active] <= 1e-6).all())
    assert bool(torch.isfinite(lse[active]).all())
    if a.mask is not None:
        off = ~active
        assert bool((lp[off] == 0).all()) and bool((lse[off] == 0).all())
        assert bool((gx[off].view(torch.int16) == 0).all()), "masked rows not +0.0"
    # every active row of the gradient sums to ~0 (softmax sums to one), up to
    # the rounding of each stored element (at most 2^-8 of it in bf16)
    ga = gx[active].double()
    rs = ga.sum(dim=1).abs()
    bound = 2.0 ** -8 * ga.abs().sum(dim=1) + 1e-5
    assert bool((rs <= bound).all())


def test_split_invariance():
    """The same rows computed under different cluster splits (chosen from N)
    agree with each other and with the oracle."""
    dev = device()
    big = W.make_logits_inputs("c151k", device=dev, N=5000)
    outs = []
    for N in (4, 600, 1000, 2000, 5000):
        x, t = big.x[:N], big.t[:N]
        lp, lse = slp.slp_forward(x, t, None, 1.0)
        torch.cuda.synchronize()
        outs.append((to64(lp[:4]), to64(lse[:4])))
    for lp, lse in outs[1:]:
        assert np.abs(lp - outs[0][0]).max() <= TOL_LP
        assert np.abs(lse - outs[0][1]).max() <= TOL_LP
    check_rows(big.x[:4], big.t[:4], None, 1.0, big.g[:4],
               *slp.slp_forward(big.x[:4], big.t[:4], None, 1.0), None, range(4))


def test_split_invariance_long_rows():
    """Rows of 1 MB (V = 524288 bf16) under every split the forward's rule
    picks for few rows: 8 CTAs per row (N = 2 and 50), 4 (N = 100), 1
    (N = 300) and 2 (N = 600, a little more than one wave).  The shared rows
    agree across the calls and with the oracle."""
    dev = device()
    big = W.make_logits_inputs("c151k", device=dev, N=600, V=524288)
    outs = []
    for N in (2, 50, 100, 300, 600):
        lp, lse = slp.slp_forward(big.x[:N], big.t[:N], None, 1.0)
        torch.cuda.synchronize()
        outs.append((to64(lp[:2]), to64(lse[:2])))
    for lp, lse in outs[1:]:
        assert np.abs(lp - outs[0][0]).max() <= TOL_LP
        assert np.abs(lse - outs[0][1]).max() <= TOL_LP
    lp, lse = slp.slp_forward(big.x[:100], big.t[:100], None, 1.0)
    check_rows(big.x[:100], big.t[:100], None, 1.0, big.g[:100], lp, lse, None, range(100))


def test_short_rows_both_forward_kernels():
    """Rows of 60 KB take the warp-per-row forward when there are many rows
    and the ring kernel when there are few; the same rows agree across the
    two and with the oracle (logits path tolerances)."""
    dev = device()
    big = W.make_logits_inputs("c151k", device=dev, N=4000, V=30000)
    lp_many, lse_many = slp.slp_forward(big.x, big.t, None, 1.0)
    lp_few, lse_few = slp.slp_forward(big.x[:1000], big.t[:1000], None, 1.0)
    torch.cuda.synchronize()
    assert float((lp_many[:1000] - lp_few).abs().max()) <= TOL_LP
    assert float((lse_many[:1000] - lse_few).abs().max()) <= TOL_LP
    rows = [0, 1, 517, 999, 1000, 3999]
    gx = slp.slp_backward(big.x, big.t, None, 1.0, lse_many, big.g)
    check_rows(big.x, big.t, None, 1.0, big.g, lp_many, lse_many, gx, rows)


def test_deterministic():
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev, N=512)
    r1 = run(a.x, a.t, a.mask, a.T, a.g)
    r2 = run(a.x, a.t, a.mask, a.T, a.g)
    for u, v in zip(r1, r2):
        assert torch.equal(u.view(torch.int16) if u.dtype == torch.bfloat16 else u.view(torch.int32),
                           v.view(torch.int16) if v.dtype == torch.bfloat16 else v.view(torch.int32))


def test_deterministic_full_size():
    """Forward and backward twice at full size (c151k), bit-identical: every
    row's ring of bulk copies is reused 4-5 times per row."""
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev)
    lp1, lse1 = slp.slp_forward(a.x, a.t, a.mask, a.T)
    lp2, lse2 = slp.slp_forward(a.x, a.t, a.mask, a.T)
    gx1 = slp.slp_backward(a.x, a.t, a.mask, a.T, lse1, a.g)
    gx2 = slp.slp_backward(a.x, a.t, a.mask, a.T, lse1, a.g)
    torch.cuda.synchronize()
    assert torch.equal(lp1.view(torch.int32), lp2.view(torch.int32))
    assert torch.equal(lse1.view(torch.int32), lse2.view(torch.int32))
    assert torch.equal(gx1.view(torch.int16), gx2.view(torch.int16))


def test_empty_and_degenerate():
    dev = device()
    # N = 0
    x = torch.empty((0, 100), dtype=torch.bfloat16, device=dev)
    t = torch.empty(0, dtype=torch.int32, device=dev)
    lp, lse = slp.slp_forward(x, t, None, 1.0)
    gx = slp.slp_backward(x, t, None, 1.0, lse, torch.empty(0, device=dev))
    assert lp.numel() == 0 and gx.shape == (0, 100)
    # V = 1: logprob 0, gradient 0
    x = torch.randn(5, 1, device=dev)
    t = torch.zeros(5, dtype=torch.int32, device=dev)
    g = torch.ones(5, device=dev)
    lp, lse, gx = run(x, t, None, 0.9, g)
    assert float(lp.abs().max()) <= TOL_LP
    assert float(gx.abs().max()) <= 1e-5
    # all-zero mask, all-one mask, mask None
    a = W.make_logits_inputs("tiny", device=dev, N=64, V=4096)
    z = torch.zeros(64, dtype=torch.uint8, device=dev)
    lp0, lse0, gx0 = run(a.x, a.t, z, a.T, a.g)
    assert bool((lp0 == 0).all()) and bool((lse0 == 0).all())
    assert bool((gx0.view(torch.int16) == 0).all())
    lp1, lse1, gx1 = run(a.x, a.t, torch.ones_like(z), a.T, a.g)
    lpn, lsen, gxn = run(a.x, a.t, None, a.T, a.g)
    assert torch.equal(lp1, lpn) and torch.equal(gx1, gxn)


def test_target_on_neg_inf_and_all_neg_inf_rows():
    dev = device()
    x = torch.randn(3, 1000, device=dev)
    x[0, 5] = float("-inf")
    x[1, :] = float("-inf")
    t = torch.tensor([5, 0, 7], dtype=torch.int32, device=dev)
    lp, lse = slp.slp_forward(x, t, None, 1.0)
    torch.cuda.synchronize()
    assert float(lp[0]) == float("-inf")
    assert np.isnan(float(lp[1])) and np.isnan(float(lse[1]))
    r, _ = O.selected_logprob_forward(to64(x[2:]), [7], None, 1.0)
    assert abs(float(lp[2]) - r[0]) <= TOL_LP


def test_bad_target_sets_error_word():
    dev = device()
    a = W.make_logits_inputs("tiny", device=dev, N=16, V=512)
    t = a.t.clone()
    t[3] = 512
    t[9] = -1
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse = slp.slp_forward(a.x, t, None, 1.0, err=err)
    gx = slp.slp_backward(a.x, t, None, 1.0, lse, a.g, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    assert np.isnan(float(lp[3])) and np.isnan(float(lp[9]))
    assert bool(torch.isnan(gx[3].float()).all())
    good = [i for i in range(16) if i not in (3, 9)]
    check_rows(a.x, t, None, 1.0, a.g, lp, lse, gx, good)
    # masked-off bad targets are not errors
    err.zero_()
    m = torch.ones(16, dtype=torch.uint8, device=dev)
    m[3] = m[9] = 0
    slp.slp_forward(a.x, t, m, 1.0, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_strided_unaligned_rows_fp32():
    dev = device()
    base = torch.randn(20, 1003, device=dev) * 3
    x = base[:, 1:1002]                  # ld = 1003 floats, rows not 16-byte aligned
    t = torch.randint(0, 1001, (20,), dtype=torch.int32, device=dev)
    g = torch.rand(20, device=dev) * 2 - 1
    lp, lse, gx = run(x, t, None, 1.3, g)
    check_rows(x, t, None, 1.3, g, lp, lse, gx, range(20))


def test_autograd_and_side_stream():
    dev = device()
    a = W.make_logits_inputs("tiny", device=dev, N=128, V=3000)
    x = a.x.clone().requires_grad_(True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lp = slp.selected_logprob(x, a.t, None, a.T)
        (lp * a.g).sum().backward()
    s.synchronize()
    _, lse = slp.slp_forward(a.x, a.t, None, a.T)
    ref = slp.slp_backward(a.x, a.t, None, a.T, lse, a.g)
    torch.cuda.synchronize()
    assert torch.equal(x.grad, ref)
    check_rows(a.x, a.t, None, a.T, a.g, lp.detach(), lse, x.grad, range(0, 128, 7))


# ---- fused forward + backward (slp_forward_backward) -------------------------

FB_SCALED = [
    ("tiny", None, None),             # 4 KB rows: one warp per row
    ("c151k", 48, 151936),            # cluster of 4
    ("c151k", 33, 151936 - 5),        # ragged tail: rows not 16-byte aligned -> separate kernels
    ("packed", 3000, 20016),
    ("stability", 256, 131072),       # fp32: 4 CTAs with the TMEM part (7 without)
    ("stability", 40, 75968),         # fp32, 4 CTAs: the TMEM part would save only one
    ("tiny", 300, 2047),              # unaligned rows -> separate kernels
]


@pytest.mark.parametrize("name,N,V", FB_SCALED, ids=lambda v: str(v))
def test_fused_forward_backward_all_rows(name, N, V):
    dev = device()
    a = W.make_logits_inputs(name, device=dev, N=N, V=V)
    lp, lse, gx = slp.slp_forward_backward(a.x, a.t, a.mask, a.T, a.g)
    torch.cuda.synchronize()
    check_rows(a.x, a.t, a.mask, a.T, a.g, lp, lse, gx, range(a.x.shape[0]))


@pytest.mark.parametrize("name", FULL)
def test_fused_forward_backward_full_size(name):
    dev = device()
    a = W.make_logits_inputs(name, device=dev)
    N = a.x.shape[0]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, gx = slp.slp_forward_backward(a.x, a.t, a.mask, a.T, a.g, err=err)
    lp2, lse2 = slp.slp_forward(a.x, a.t, a.mask, a.T, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0  # no data error and no wait that gave up
    rows = set(np.random.default_rng(23).choice(N, 24, replace=False).tolist()) | {0, N - 1}
    check_rows(a.x, a.t, a.mask, a.T, a.g, lp, lse, gx, rows)
    # same quantity as the separate forward, every row
    assert float((lp - lp2).abs().max()) <= TOL_LP and float((lse - lse2).abs().max()) <= TOL_LP
    if a.mask is not None:
        off = a.mask == 0
        assert bool((gx[off].view(torch.int16) == 0).all())


def test_fused_forward_backward_deterministic_full_size():
    """The fused call twice on c151k at full size (clusters of 4 CTAs per row,
    merged through distributed shared memory), bit-identical."""
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev)
    r1 = slp.slp_forward_backward(a.x, a.t, a.mask, a.T, a.g)
    r2 = slp.slp_forward_backward(a.x, a.t, a.mask, a.T, a.g)
    torch.cuda.synchronize()
    assert torch.equal(r1[0].view(torch.int32), r2[0].view(torch.int32))
    assert torch.equal(r1[1].view(torch.int32), r2[1].view(torch.int32))
    assert torch.equal(r1[2].view(torch.int16), r2[2].view(torch.int16))


@pytest.mark.parametrize("name,V,Vp", [("tiny", 350000, 350000), ("tiny", 349997, 350000),
                                       ("stability", 175000, 175000), ("tiny", 400008, 400008),
                                       ("tiny", 560000, 560000)])
def test_fused_forward_backward_tmem_long_rows(name, V, Vp):
    """Rows of 700 KB to 1.09 MB: longer than eight CTAs of the register form
    hold, so the cluster kernel runs its TMEM form (5 to 8 CTAs per row); one
    bf16 case with a scalar tail on an aligned stride, one fp32 case."""
    dev = device()
    a = W.make_logits_inputs(name, device=dev, N=6, V=Vp)
    x = a.x[:, :V]
    t = a.t % V
    t[0] = V - 1
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, gx = slp.slp_forward_backward(x, t, None, a.T, a.g, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_rows(x, t, None, a.T, a.g, lp, lse, gx, range(6))


@pytest.mark.parametrize("V", [600000, 620008])
def test_fused_forward_backward_long_rows(V):
    """Rows longer than one cluster holds (8 CTAs of the TMEM form, about
    1.1 MB) take the separate kernels and still match the oracle."""
    dev = device()
    a = W.make_logits_inputs("tiny", device=dev, N=5, V=V)
    lp, lse, gx = slp.slp_forward_backward(a.x, a.t, a.mask, a.T, a.g)
    torch.cuda.synchronize()
    check_rows(a.x, a.t, a.mask, a.T, a.g, lp, lse, gx, range(5))


# Short rows (at most 32 KB) take the warp-per-row fused kernel: V chosen so
# that each register width (1, 2, 4, 8, 16 vectors per lane) and the
# shared-memory slot (rows above 8 KB) is used, some with a scalar tail.
FB_ROWS = [
    ("packed", 70, 200),        # bf16, 1 vector per lane, masked spans
    ("tiny", 37, 504),          # 2 per lane
    ("packed", 65, 1000),       # 4 per lane
    ("tiny", 33, 4096),         # 16 per lane, all in registers
    ("c151k", 41, 4104),        # 16 per lane + one vector per lane in shared memory
    ("c151k", 64, 8192),        # 8 KB in registers, 8 KB in shared memory
    ("packed", 300, 16384),     # the longest row: 8 KB + 24 KB
    ("stability", 29, 2048),    # fp32, 16 per lane, inf/-inf rows
    ("stability", 22, 8192),    # fp32, 32 KB
]


@pytest.mark.parametrize("name,N,V", FB_ROWS, ids=lambda v: str(v))
def test_fused_short_rows_all_rows(name, N, V):
    dev = device()
    a = W.make_logits_inputs(name, device=dev, N=N, V=V)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, gx = slp.slp_forward_backward(a.x, a.t, a.mask, a.T, a.g, err=err)
    lp2, lse2 = slp.slp_forward(a.x, a.t, a.mask, a.T)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_rows(a.x, a.t, a.mask, a.T, a.g, lp, lse, gx, range(N))
    assert_close_nan(to64(lp), to64(lp2), TOL_LP, "logprob vs separate forward")
    if a.mask is not None:
        assert bool((gx[a.mask == 0].view(torch.int16 if gx.dtype == torch.bfloat16
                                          else torch.int32) == 0).all())


@pytest.mark.parametrize("V", [4101, 16381])
def test_fused_short_rows_ragged_tail(V):
    """Rows of V not a multiple of 8 on a 16-byte-aligned stride: the scalar
    tail of the warp-per-row kernel, targets in the tail included, and
    grad_x's padding columns left untouched."""
    dev = device()
    Vp = (V + 7) // 8 * 8
    a = W.make_logits_inputs("c151k", device=dev, N=48, V=Vp)
    x = a.x[:, :V]
    t = a.t % V
    t[:8] = V - 1 - torch.arange(8, dtype=torch.int32, device=dev) % (V % 8)
    gx = torch.full((48, Vp), 7.0, dtype=torch.bfloat16, device=dev)
    lp, lse, _ = slp.slp_forward_backward(x, t, None, a.T, a.g, grad_x=gx[:, :V])
    torch.cuda.synchronize()
    assert bool((gx[:, V:] == 7.0).all())
    check_rows(x, t, None, a.T, a.g, lp, lse, gx[:, :V], range(48))


@pytest.mark.parametrize("V,Vp", [(65536, 65536), (100000, 100000), (150000, 150000),
                                  (100001, 100004)])
def test_fused_tmem_form_fp32_rows(V, Vp):
    """fp32 rows for which the fused call keeps part of each segment in TMEM
    (2, 3, 5 and 3 CTAs per row instead of 4, 6, 8 and 6; the last with a
    scalar tail of one element on a padded row stride): every row against the
    oracle, with two masked rows and one bad target, then the same call again
    bit for bit."""
    dev = device()
    a = W.make_logits_inputs("stability", device=dev, N=20, V=Vp)
    x = a.x[:, :V]
    mask = torch.ones(20, dtype=torch.uint8, device=dev)
    mask[3] = 0
    mask[11] = 0
    t = a.t % V
    t[7] = V + 5
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # gradients on the same padded stride, so both row sets stay 16-byte aligned
    gx = torch.empty((20, Vp), dtype=x.dtype, device=dev)[:, :V]
    gx2 = torch.empty((20, Vp), dtype=x.dtype, device=dev)[:, :V]
    lp, lse, _ = slp.slp_forward_backward(x, t, mask, a.T, a.g, grad_x=gx, err=err)
    lp2, lse2, _ = slp.slp_forward_backward(x, t, mask, a.T, a.g, grad_x=gx2)
    torch.cuda.synchronize()
    assert int(err.item()) == 1  # the bad target's data error, nothing else
    assert np.isnan(float(lp[7])) and bool(torch.isnan(gx[7]).all())
    check_rows(x, t, mask, a.T, a.g, lp, lse, gx, [r for r in range(20) if r != 7])
    assert torch.equal(lp.view(torch.int32), lp2.view(torch.int32))
    assert torch.equal(gx.view(torch.int32), gx2.view(torch.int32))


def test_fused_forward_backward_bad_target():
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev, N=8, V=151936)
    t = a.t.clone()
    t[2] = -5
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, gx = slp.slp_forward_backward(a.x, t, None, 1.0, a.g, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    assert np.isnan(float(lp[2])) and bool(torch.isnan(gx[2].float()).all())
    check_rows(a.x, t, None, 1.0, a.g, lp, lse, gx, [0, 1, 3, 4, 5, 6, 7])


def test_fused_short_rows_bad_target():
    """A bad target on the warp-per-row fused kernel: the error bit, NaN
    logprob, lse and gradient for that row, the other rows exact to the
    oracle."""
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev, N=40, V=8192)
    t = a.t.clone()
    t[5] = 8192
    t[17] = -3
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, gx = slp.slp_forward_backward(a.x, t, None, 1.0, a.g, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    for r in (5, 17):
        assert np.isnan(float(lp[r])) and bool(torch.isnan(gx[r].float()).all())
    good = [i for i in range(40) if i not in (5, 17)]
    check_rows(a.x, t, None, 1.0, a.g, lp, lse, gx, good)


@pytest.mark.parametrize("V,dtype", [(1, torch.bfloat16), (3, torch.bfloat16), (7, torch.bfloat16),
                                     (1, torch.float32), (3, torch.float32)])
def test_rows_shorter_than_one_vector(V, dtype):
    """Rows of fewer elements than one 16-byte vector on an aligned stride:
    every warp-per-row kernel runs its scalar tail only (forward, backward,
    fused, entropy); the padding columns stay untouched."""
    dev = device()
    ld = 16 // (2 if dtype == torch.bfloat16 else 4)
    N = 50
    gen = torch.Generator(device=dev).manual_seed(5)
    full = (torch.randn((N, ld), generator=gen, device=dev) * 3).to(dtype)
    x = full[:, :V]
    t = torch.randint(0, V, (N,), generator=gen, device=dev, dtype=torch.int32)
    g = torch.rand(N, generator=gen, device=dev) * 2 - 1
    mask = (torch.arange(N, device=dev) % 4 != 1).to(torch.uint8)
    for T in (1.0, 0.6):
        gx = torch.full((N, ld), 7.0, dtype=dtype, device=dev)
        lp, lse = slp.slp_forward(x, t, mask, T)
        slp.slp_backward(x, t, mask, T, lse, g, grad_x=gx[:, :V])
        gxf = torch.full((N, ld), 7.0, dtype=dtype, device=dev)
        lpf, lsef, _ = slp.slp_forward_backward(x, t, mask, T, g, grad_x=gxf[:, :V])
        lpe, lsee, H = slp.slp_forward_entropy(x, t, mask, T)
        torch.cuda.synchronize()
        assert bool((gx[:, V:] == 7.0).all()) and bool((gxf[:, V:] == 7.0).all())
        # the fp32 lse floor: at V = 1 the exact gradient is 0 and 1 - p is
        # one ulp of |x/T| + |lse| (x here reaches ~10)
        check_rows(x, t, mask, T, g, lp, lse, gx[:, :V], range(N), fp32_floor=True)
        check_rows(x, t, mask, T, g, lpf, lsef, gxf[:, :V], range(N), fp32_floor=True)
        assert float((lpe - lp).abs().max()) <= TOL_LP
        if V == 1:
            act = mask != 0
            assert bool((lp[act].abs() <= TOL_LP).all()) and bool((H[act].abs() <= 1e-5).all())


def test_fused_forward_backward_ragged_tail():
    """V not a multiple of 8 with a 16-byte-aligned stride: the cluster path's
    scalar tail, and grad_x's padding columns left untouched."""
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev, N=40, V=20016)
    V = 20011
    x = a.x[:, :V]
    gx = torch.full((40, 20016), 7.0, dtype=torch.bfloat16, device=dev)
    lp, lse, _ = slp.slp_forward_backward(x, a.t % V, None, a.T, a.g, grad_x=gx[:, :V])
    torch.cuda.synchronize()
    assert bool((gx[:, V:] == 7.0).all())
    check_rows(x, a.t % V, None, a.T, a.g, lp, lse, gx[:, :V], range(40))
