"""GPU parity of the top-k forward KL (slp_topk_kl_forward / _backward)
against the CPU oracle.

Tolerances: kl, student_mass, teacher_mass within 5e-5 absolute (sums of K
fp32 terms built on an lse carrying ~1e-5); lse within 2e-5; gradients
within 2^-8 |ref| + 1e-6 per element (the logits-path bound)."""

import numpy as np
import pytest
import torch

import vocab_selected_token_gb300 as slp
from oracle import slp_oracle as O
from tests.gpu_util import assert_close_nan, assert_grad_close, device, to64
from vocab_selected_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TOL = 5e-5


def check(a, kl, sm, tm, lse, gx, rows, clamp):
    rows = np.asarray(sorted(set(int(r) for r in rows)))
    ridx = torch.as_tensor(rows, device=a.x.device)
    x64 = to64(a.x[ridx])
    ids = a.ids[ridx].cpu().numpy()
    lt = to64(a.lt[ridx])
    m = None if a.mask is None else a.mask[ridx].cpu().numpy()
    cl = None if clamp == float("-inf") else clamp
    rkl, rsm, rtm, rlse = O.topk_kl_forward(x64, ids, lt, m, a.T, cl)
    assert_close_nan(to64(lse[ridx]), rlse, 2e-5, "lse")
    assert_close_nan(to64(kl[ridx]), rkl, TOL, "kl")
    assert_close_nan(to64(sm[ridx]), rsm, TOL, "student mass")
    assert_close_nan(to64(tm[ridx]), rtm, TOL, "teacher mass")
    if gx is not None:
        rgx = O.topk_kl_backward(x64, ids, lt, m, a.T, cl, rlse, to64(a.g[ridx]))
        assert_grad_close(to64(gx[ridx]), rgx, "top-k kl grad")


def run(a, clamp):
    kl, sm, tm, lse = slp.slp_topk_kl_forward(a.x, a.ids, a.lt, a.mask, a.T, clamp)
    gx = slp.slp_topk_kl_backward(a.x, a.ids, a.lt, a.mask, a.T, clamp, lse, a.g)
    torch.cuda.synchronize()
    return kl, sm, tm, lse, gx


# (192, 2048, 32) and (64, 20016, 128) take the warp-per-row backward, the
# others one CTA per row (unaligned rows, a 297 KB row, K above 256).
CASES = [(192, 2048, 32), (64, 20016, 128), (33, 2047, 16), (40, 151936, 64),
         (24, 4096, 300)]


@pytest.mark.parametrize("N,V,K", CASES, ids=lambda v: str(v))
@pytest.mark.parametrize("clamp", [float("-inf"), -10.0])
def test_topk_all_rows(N, V, K, clamp):
    dev = device()
    a = W.make_topk_inputs(device=dev, N=N, V=V, K=K)
    out = run(a, clamp)
    check(a, *out, range(N), clamp)


def test_topk_fp32_masked_repeated_ids():
    dev = device()
    a = W.make_topk_inputs(device=dev, N=50, V=4096, K=24)
    a.x = a.x.float() * 1.5
    a.ids[:, 5] = a.ids[:, 3]                 # a repeated id in every row
    a.mask = (torch.arange(50, device=dev) % 3 != 0).to(torch.uint8)
    kl, sm, tm, lse, gx = run(a, -10.0)
    check(a, kl, sm, tm, lse, gx, range(50), -10.0)
    off = a.mask == 0
    assert bool((kl[off] == 0).all()) and bool((gx[off].view(torch.int32) == 0).all())


def test_topk_full_size_sampled():
    dev = device()
    a = W.make_topk_inputs(device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kl, sm, tm, lse = slp.slp_topk_kl_forward(a.x, a.ids, a.lt, a.mask, a.T, a.clamp, err=err)
    gx = slp.slp_topk_kl_backward(a.x, a.ids, a.lt, a.mask, a.T, a.clamp, lse, a.g, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0  # no data error and no wait that gave up
    N = a.x.shape[0]
    rows = set(np.random.default_rng(31).choice(N, 16, replace=False).tolist()) | {0, N - 1}
    check(a, kl, sm, tm, lse, gx, rows, a.clamp)
    assert bool(torch.isfinite(kl).all()) and bool(torch.isfinite(gx.float()).all())


def test_topk_bad_id_flagged():
    dev = device()
    a = W.make_topk_inputs(device=dev, N=8, V=3000, K=8)
    a.ids[2, 4] = 3000
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kl, sm, tm, lse = slp.slp_topk_kl_forward(a.x, a.ids, a.lt, None, a.T, -10.0, err=err)
    gx = slp.slp_topk_kl_backward(a.x, a.ids, a.lt, None, a.T, -10.0, lse, a.g, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    assert np.isnan(float(kl[2])) and bool(torch.isnan(gx[2].float()).all())
    check(a, kl, sm, tm, lse, gx, [0, 1, 3, 4, 5, 6, 7], -10.0)


def test_topk_short_rows_ragged_tail():
    """Warp-per-row backward on rows whose V is not a multiple of 8 (16-byte
    aligned stride): ids in the scalar tail, repeated ids from the wrap, and
    grad_x's padding columns left untouched."""
    dev = device()
    V, Vp = 4101, 4104
    a = W.make_topk_inputs(device=dev, N=40, V=Vp, K=32)
    a.x = a.x[:, :V]
    a.ids = a.ids % V
    a.ids[:, 0] = V - 1
    a.ids[:, 1] = V - 4
    kl, sm, tm, lse = slp.slp_topk_kl_forward(a.x, a.ids, a.lt, None, a.T, -10.0)
    gx = torch.full((40, Vp), 7.0, dtype=torch.bfloat16, device=dev)
    slp.slp_topk_kl_backward(a.x, a.ids, a.lt, None, a.T, -10.0, lse, a.g, grad_x=gx[:, :V])
    torch.cuda.synchronize()
    assert bool((gx[:, V:] == 7.0).all())
    check(a, kl, sm, tm, lse, gx[:, :V], range(40), -10.0)


def test_topk_backward_deterministic_full_size():
    """Three backward runs at full size are bit-identical.  Guards the ring of
    the CTA-per-row kernel: each thread fences its shared-memory reads of a
    stage against the bulk copy that refills it (without the fence a read
    still queued behind the kernel's own stores could return the next
    chunk's bytes in a few rows per run)."""
    dev = device()
    a = W.make_topk_inputs(device=dev)
    kl, sm, tm, lse = slp.slp_topk_kl_forward(a.x, a.ids, a.lt, a.mask, a.T, a.clamp)
    first = slp.slp_topk_kl_backward(a.x, a.ids, a.lt, a.mask, a.T, a.clamp, lse, a.g)
    for _ in range(2):
        again = slp.slp_topk_kl_backward(a.x, a.ids, a.lt, a.mask, a.T, a.clamp, lse, a.g)
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))
        del again


def test_topk_rows_shorter_than_one_vector():
    """V = 7 on a 16-byte stride (bf16): the warp-per-row backward runs its
    scalar tail only; K = 3 with a repeated id in half of the rows."""
    dev = device()
    a = W.make_topk_inputs(device=dev, N=30, V=8, K=3)
    V = 7
    a.x = a.x[:, :V]
    a.ids = a.ids % V
    a.ids[::2, 2] = a.ids[::2, 0]
    kl, sm, tm, lse = slp.slp_topk_kl_forward(a.x, a.ids, a.lt, None, a.T, -10.0)
    gx = torch.full((30, 8), 7.0, dtype=torch.bfloat16, device=dev)
    slp.slp_topk_kl_backward(a.x, a.ids, a.lt, None, a.T, -10.0, lse, a.g, grad_x=gx[:, :V])
    torch.cuda.synchronize()
    assert bool((gx[:, V:] == 7.0).all())
    check(a, kl, sm, tm, lse, gx[:, :V], range(30), -10.0)
