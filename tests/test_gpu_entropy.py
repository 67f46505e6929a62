"""GPU parity of slp_forward_entropy / slp_backward_entropy (per-token entropy
in the same pass) against the CPU oracle.

Entropy tolerance: |dH| <= 5e-5 + 1e-5 |H|.  H = ln s - (w/s)/T is formed in
fp32 from two accumulated sums; each carries ~1e-6 relative error (ex2.approx
plus fp32 adds over up to 2.5e5 terms) on terms of magnitude up to ~20, so a
few 1e-5 absolute is the fp32 floor.  logprob/lse and gradients use the
logits-path tolerances."""

import numpy as np
import pytest
import torch

import vocab_selected_token_gb300 as slp
from oracle import slp_oracle as O
from tests.gpu_util import TOL_LP, assert_close_nan, assert_grad_close, device, to64
from vocab_selected_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def check_entropy_rows(a, gH, lp, lse, H, gx, rows):
    rows = np.asarray(sorted(set(int(r) for r in rows)))
    ridx = torch.as_tensor(rows, device=a.x.device)
    x64 = to64(a.x[ridx])
    t = a.t[ridx].cpu().numpy()
    m = None if a.mask is None else a.mask[ridx].cpu().numpy()
    rlp, rlse, rH = O.entropy_forward(x64, t, m, a.T)
    assert_close_nan(to64(lp[ridx]), rlp, TOL_LP, "logprob")
    assert_close_nan(to64(lse[ridx]), rlse, TOL_LP, "lse")
    Hg = to64(H[ridx])
    fin = np.isfinite(rH)
    assert (np.isfinite(Hg) == fin).all()
    err = np.abs(Hg[fin] - rH[fin])
    assert (err <= 5e-5 + 1e-5 * np.abs(rH[fin])).all(), f"entropy max err {err.max():.2e}"
    if gx is not None:
        rgx = O.entropy_backward(x64, t, m, a.T, rlse, rH, to64(a.g[ridx]), to64(gH[ridx]))
        assert_grad_close(to64(gx[ridx]), rgx, "entropy grad")


CASES = [("tiny", None, None), ("c151k", 48, 151936), ("packed", 3000, 20016),
         ("stability", 256, 131072), ("tiny", 300, 2047), ("c151k", 6, 151936),
         ("stability", 40, 3000), ("packed", 90, 600)]


@pytest.mark.parametrize("name,N,V", CASES, ids=lambda v: str(v))
def test_entropy_all_rows(name, N, V):
    dev = device()
    a = W.make_logits_inputs(name, device=dev, N=N, V=V)
    gH = torch.rand(a.x.shape[0], device=dev) * 2 - 1
    lp, lse, H = slp.slp_forward_entropy(a.x, a.t, a.mask, a.T)
    gx = slp.slp_backward_entropy(a.x, a.t, a.mask, a.T, lse, H, a.g, gH)
    torch.cuda.synchronize()
    check_entropy_rows(a, gH, lp, lse, H, gx, range(a.x.shape[0]))
    if a.mask is not None:
        off = a.mask == 0
        assert bool((H[off] == 0).all()) and bool((gx[off].view(torch.int16) == 0).all())


@pytest.mark.parametrize("name", ["c151k", "packed", "stability"])
def test_entropy_full_size_sampled(name):
    dev = device()
    a = W.make_logits_inputs(name, device=dev)
    N = a.x.shape[0]
    gH = torch.rand(N, device=dev) * 2 - 1
    lp, lse, H = slp.slp_forward_entropy(a.x, a.t, a.mask, a.T)
    gx = slp.slp_backward_entropy(a.x, a.t, a.mask, a.T, lse, H, a.g, gH)
    lp0, lse0 = slp.slp_forward(a.x, a.t, a.mask, a.T)
    torch.cuda.synchronize()
    rows = set(np.random.default_rng(29).choice(N, 24, replace=False).tolist()) | {0, N - 1}
    if name == "stability":
        rows |= set(torch.nonzero(torch.isinf(a.x).any(dim=1))[:4, 0].tolist())
    check_entropy_rows(a, gH, lp, lse, H, gx, rows)
    assert torch.equal(lp, lp0) or float((lp - lp0).abs().max()) <= TOL_LP
    act = torch.ones(N, dtype=torch.bool, device=dev) if a.mask is None else a.mask != 0
    assert bool(torch.isfinite(H[act]).all()) and bool((H[act] >= -1e-4).all())


def test_entropy_gradient_parts():
    """grad_entropy = NULL is the plain backward, bit for bit; grad_out = NULL
    leaves only the entropy term."""
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev, N=64)
    lp, lse, H = slp.slp_forward_entropy(a.x, a.t, None, 1.0)
    g_only = slp.slp_backward_entropy(a.x, a.t, None, 1.0, lse, H, a.g, None)
    plain = slp.slp_backward(a.x, a.t, None, 1.0, lse, a.g)
    gH = torch.rand(64, device=dev)
    h_only = slp.slp_backward_entropy(a.x, a.t, None, 1.0, lse, H, None, gH)
    torch.cuda.synchronize()
    assert torch.equal(g_only, plain)
    zero_g = torch.zeros_like(a.g)
    rlp, rlse, rH = O.entropy_forward(to64(a.x), a.t.cpu().numpy(), None, 1.0)
    ref = O.entropy_backward(to64(a.x), a.t.cpu().numpy(), None, 1.0, rlse, rH, to64(zero_g),
                             to64(gH))
    assert_grad_close(to64(h_only), ref, "entropy-only gradient")


def test_entropy_autograd():
    dev = device()
    a = W.make_logits_inputs("tiny", device=dev, N=64, V=5000)
    x = a.x.clone().requires_grad_(True)
    gH = torch.rand(64, device=dev)
    lp, H = slp.selected_logprob_and_entropy(x, a.t, None, a.T)
    ((lp * a.g).sum() + (H * gH).sum()).backward()
    _, lse, H2 = slp.slp_forward_entropy(a.x, a.t, None, a.T)
    ref = slp.slp_backward_entropy(a.x, a.t, None, a.T, lse, H2, a.g, gH)
    torch.cuda.synchronize()
    assert torch.equal(x.grad, ref)


# ---- fused forward + backward with the entropy (slp_forward_backward_entropy) ----

FB_ENT = [
    ("tiny", None, None),          # 4 KB rows: one warp per row
    ("packed", 90, 600),           # short rows with masked spans
    ("stability", 40, 3000),       # fp32 short rows
    ("c151k", 48, 151936),         # cluster of 4 CTAs per row
    ("packed", 300, 20016),        # 40 KB rows: cluster
    ("stability", 256, 131072),    # fp32, rows with -inf columns; TMEM part, 4 CTAs
    ("stability", 24, 65536),      # fp32, TMEM part: 2 CTAs per row instead of 4
    ("stability", 16, 150000),     # fp32, TMEM part: 5 CTAs per row instead of 8
    ("tiny", 300, 2047),           # unaligned rows: the separate kernels
]


@pytest.mark.parametrize("name,N,V", FB_ENT, ids=lambda v: str(v))
def test_fused_entropy_all_rows(name, N, V):
    dev = device()
    a = W.make_logits_inputs(name, device=dev, N=N, V=V)
    gH = torch.rand(a.x.shape[0], device=dev) * 2 - 1
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, H, gx = slp.slp_forward_backward_entropy(a.x, a.t, a.mask, a.T, a.g, gH, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_entropy_rows(a, gH, lp, lse, H, gx, range(a.x.shape[0]))
    if a.mask is not None:
        off = a.mask == 0
        zero = gx[off].view(torch.int16 if gx.dtype == torch.bfloat16 else torch.int32) == 0
        assert bool((H[off] == 0).all()) and bool(zero.all())


def test_fused_entropy_full_size():
    """c151k at full size: sampled rows against the oracle, and every row's
    logprob, lse and entropy against the separate entropy forward."""
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev)
    N = a.x.shape[0]
    gH = torch.rand(N, device=dev) * 2 - 1
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, H, gx = slp.slp_forward_backward_entropy(a.x, a.t, a.mask, a.T, a.g, gH, err=err)
    lp2, lse2, H2 = slp.slp_forward_entropy(a.x, a.t, a.mask, a.T)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = set(np.random.default_rng(41).choice(N, 20, replace=False).tolist()) | {0, N - 1}
    check_entropy_rows(a, gH, lp, lse, H, gx, rows)
    assert float((lp - lp2).abs().max()) <= TOL_LP and float((lse - lse2).abs().max()) <= TOL_LP
    assert float((H - H2).abs().max()) <= 5e-5 + 1e-5 * float(H2.abs().max())


@pytest.mark.parametrize("V", [4096, 151936])
def test_fused_entropy_null_weights(V):
    """grad_entropy = NULL leaves the plain gradient; grad_out = NULL leaves
    only the entropy term (both against the oracle)."""
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev, N=40, V=V)
    lp, lse, H, gx = slp.slp_forward_backward_entropy(a.x, a.t, None, 1.0, a.g, None)
    torch.cuda.synchronize()
    check_entropy_rows(a, torch.zeros_like(a.g), lp, lse, H, gx, range(40))
    gH = torch.rand(40, device=dev)
    lp, lse, H, gx = slp.slp_forward_backward_entropy(a.x, a.t, None, 1.0, None, gH)
    torch.cuda.synchronize()
    a.g = torch.zeros_like(a.g)
    check_entropy_rows(a, gH, lp, lse, H, gx, range(40))


@pytest.mark.parametrize("name,V", [("tiny", 350000), ("stability", 175000), ("tiny", 560000)])
def test_fused_entropy_tmem_long_rows(name, V):
    """Rows of 700 KB to 1.09 MB (bf16 and fp32): the cluster kernel's TMEM
    form with the entropy."""
    dev = device()
    a = W.make_logits_inputs(name, device=dev, N=6, V=V)
    gH = torch.rand(6, device=dev) * 2 - 1
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, H, gx = slp.slp_forward_backward_entropy(a.x, a.t, None, a.T, a.g, gH, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_entropy_rows(a, gH, lp, lse, H, gx, range(6))


@pytest.mark.parametrize("V", [8192, 151936])
def test_fused_entropy_bad_target(V):
    dev = device()
    a = W.make_logits_inputs("c151k", device=dev, N=24, V=V)
    t = a.t.clone()
    t[3] = V
    t[11] = -2
    a.t = t
    gH = torch.rand(24, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, H, gx = slp.slp_forward_backward_entropy(a.x, t, None, 1.0, a.g, gH, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    for r in (3, 11):
        assert np.isnan(float(lp[r])) and np.isnan(float(H[r]))
        assert bool(torch.isnan(gx[r].float()).all())
    check_entropy_rows(a, gH, lp, lse, H, gx, [i for i in range(24) if i not in (3, 11)])
