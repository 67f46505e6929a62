"""GPU parity of the fused LM-head path (slp_lmhead_forward / _backward through
the C ABI) against the CPU oracle.

Tolerances: |logprob - oracle| <= 5e-3; gradients reach cosine >= 0.999 and
relative Frobenius error <= 1e-2 against the fp64 oracle; masked rows of dh
are exactly +0.0."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import vocab_selected_token_gb300 as slp
from oracle import slp_oracle as O
from tests.gpu_util import assert_close_nan, device, to64
from vocab_selected_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_LP = 5e-3
COS_MIN = 0.999
FROB_MAX = 1e-2


def grad_ok(got, ref, what):
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    nr = np.linalg.norm(ref)
    if nr == 0:
        assert np.all(got == 0), f"{what}: expected all zeros"
        return
    cos = float(got @ ref / (np.linalg.norm(got) * nr + 1e-300))
    frob = float(np.linalg.norm(got - ref) / nr)
    assert cos >= COS_MIN and frob <= FROB_MAX, f"{what}: cosine {cos:.6f} frob {frob:.3e}"


def run_fwd_bwd(a, err=None):
    lp, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T, err=err)
    dh, dW = slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, lse, a.g, err=err)
    torch.cuda.synchronize()
    return lp, lse, dh, dW


SMALL = [
    # N, V, d, T, p_mask
    (300, 1000, 128, 1.0, 0.5),     # ragged row block and vocabulary tile
    (256, 512, 64, 0.7, 1.0),       # one k-block, all rows active
    (1024, 20000, 512, 0.8, 0.5),   # many slabs
    (130, 4096, 2560, 1.0, 0.9),    # the workload's hidden size
]


@pytest.mark.parametrize("N,V,d,T,pm", SMALL, ids=lambda v: str(v))
def test_small_all_outputs(N, V, d, T, pm):
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=N, V=V, d=d, p_mask=pm)
    a.T = T
    lp, lse, dh, dW = run_fwd_bwd(a)
    h64, W64 = to64(a.h), to64(a.W)
    t, m, g = a.t.cpu().numpy(), a.mask.cpu().numpy(), to64(a.g)
    rlp, rlse = O.lmhead_forward(h64, W64, t, m, T)
    assert_close_nan(to64(lp), rlp, TOL_LP, "logprob")
    assert_close_nan(to64(lse), rlse, TOL_LP, "lse")
    rdh, rdW = O.lmhead_backward(h64, W64, t, m, T, rlse, g)
    grad_ok(to64(dh), rdh, "dh")
    grad_ok(to64(dW), rdW, "dW")
    off = torch.as_tensor(m == 0, device=dev)
    assert bool((dh[off].view(torch.int16) == 0).all()), "masked dh rows not +0.0"
    assert bool((lp[off] == 0).all()) and bool((lse[off] == 0).all())


def grad_rows_ok(got, ref, what):
    """grad_ok on every row on its own (an all-zero reference row must come
    back all zeros), then on the rows pooled."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    for k in range(ref.shape[0]):
        grad_ok(got[k], ref[k], f"{what}, row {k} of the sample")
    grad_ok(got, ref, f"{what} (pooled)")


def test_full_size_sampled():
    """The lmhead workload at full size (N=8192, V=151936, d=2560): logprob of
    every row, 128 rows of dh (120 active, 8 masked) and 256 rows of dW (the
    targets of the sampled active rows, the first and last vocabulary rows,
    the rest uniform) against the oracle, each row checked on its own."""
    dev = device()
    a = W.make_lmhead_inputs(device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, dh, dW = run_fwd_bwd(a, err=err)
    assert int(err.item()) == 0  # no data error and no pipeline wait that gave up
    h64, W64 = to64(a.h), to64(a.W)
    t, m, g = a.t.cpu().numpy(), a.mask.cpu().numpy(), to64(a.g)
    act = np.nonzero(m)[0]
    off_rows = np.nonzero(m == 0)[0]
    gen = np.random.default_rng(5)
    rows = sorted(set(gen.choice(act, 118, replace=False).tolist()) | {int(act[0]), int(act[-1])})
    rows += sorted(gen.choice(off_rows, 8, replace=False).tolist())
    assert len(rows) == 128
    # oracle forward for every active row (dW needs every row's lse)
    rlp, rlse = O.lmhead_forward(h64, W64, t, m, a.T)
    assert_close_nan(to64(lp), rlp, TOL_LP, "logprob (all rows)")
    rdh = O.lmhead_dh_rows(h64, W64, t, m, a.T, rlse, g, rows)
    grad_rows_ok(to64(dh[rows]), rdh, "dh")
    V = a.W.shape[0]
    vset = {int(t[r]) for r in rows if m[r]} | {0, V - 1}
    while len(vset) < 256:
        vset.add(int(gen.integers(0, V)))
    vrows = sorted(vset)
    rdW = O.lmhead_dW_rows(h64, W64, t, m, a.T, rlse, g, vrows)
    grad_rows_ok(to64(dW[vrows]), rdW, "dW")
    off = torch.as_tensor(m == 0, device=dev)
    assert bool((dh[off].view(torch.int16) == 0).all())
    assert bool(torch.isfinite(dW.float()).all()) and bool(torch.isfinite(dh.float()).all())


def test_no_mask_and_all_masked():
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=200, V=3000, d=256)
    # mask None == all-one mask
    lp1, lse1 = slp.slp_lmhead_forward(a.h, a.W, a.t, None, a.T)
    lp2, lse2 = slp.slp_lmhead_forward(a.h, a.W, a.t, torch.ones_like(a.mask), a.T)
    torch.cuda.synchronize()
    assert torch.equal(lp1, lp2) and torch.equal(lse1, lse2)
    # nothing active: zeros everywhere, dW fully overwritten with zeros
    z = torch.zeros_like(a.mask)
    lp, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, z, a.T)
    dh = torch.full((200, 256), 3.0, dtype=torch.bfloat16, device=dev)
    dW = torch.full((3000, 256), 3.0, dtype=torch.bfloat16, device=dev)
    slp.slp_lmhead_backward(a.h, a.W, a.t, z, a.T, lse, a.g, dh=dh, dW=dW)
    torch.cuda.synchronize()
    assert bool((lp == 0).all()) and bool((lse == 0).all())
    assert bool((dh.view(torch.int16) == 0).all()) and bool((dW.view(torch.int16) == 0).all())


def test_bad_target_flagged():
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=64, V=1000, d=128, p_mask=1.0)
    a.t[5] = 1000
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, dh, dW = run_fwd_bwd(a, err=err)
    assert int(err.item()) & 1
    assert np.isnan(float(lp[5])) and bool(torch.isnan(dh[5].float()).all())
    good = [i for i in range(64) if i != 5]
    m = np.ones(64, np.uint8)
    m[5] = 0  # the flagged row contributes nothing: same as masking it out
    rlp, rlse = O.lmhead_forward(to64(a.h), to64(a.W), a.t.cpu().numpy(), m, a.T)
    assert_close_nan(to64(lp[good]), rlp[good], TOL_LP, "logprob")
    _, rdW = O.lmhead_backward(to64(a.h), to64(a.W), a.t.cpu().numpy(), m, a.T, rlse, to64(a.g))
    grad_ok(to64(dW), rdW, "dW without the flagged row")


def test_deterministic():
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=700, V=9000, d=256)
    r1 = run_fwd_bwd(a)
    r2 = run_fwd_bwd(a)
    for u, v in zip(r1, r2):
        assert torch.equal(u, v)


def test_deterministic_full_size():
    """Forward and backward twice on the full lmhead workload (3 vocabulary
    chunks, split-K dh folded in order), bit-identical."""
    dev = device()
    a = W.make_lmhead_inputs(device=dev)
    r1 = run_fwd_bwd(a)
    r2 = run_fwd_bwd(a)
    for u, v in zip(r1, r2):
        assert torch.equal(u.view(torch.int16) if u.dtype == torch.bfloat16 else u.view(torch.int32),
                           v.view(torch.int16) if v.dtype == torch.bfloat16 else v.view(torch.int32))


def test_autograd():
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=128, V=2000, d=128)
    h = a.h.clone().requires_grad_(True)
    Wt = a.W.clone().requires_grad_(True)
    lp = slp.lmhead_selected_logprob(h, Wt, a.t, a.mask, a.T)
    (lp * a.g).sum().backward()
    lp2, lse2, dh, dW = run_fwd_bwd(a)
    assert torch.equal(lp.detach(), lp2)
    assert torch.equal(h.grad, dh) and torch.equal(Wt.grad, dW)


def test_backward_accumulate_into_fp32_dW():
    """Two micro-batches accumulated into one fp32 dW equal the sum of their
    oracle gradients; dh is the plain backward's, bit for bit."""
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=300, V=5000, d=256, seed=41)
    b = W.make_lmhead_inputs(device=dev, N=200, V=5000, d=256, seed=42)
    b.W = a.W  # same weights, two micro-batches
    acc = torch.randn((5000, 256), device=dev) * 1e-3
    acc0 = acc.clone()
    refs = []
    for m in (a, b):
        lp, lse = slp.slp_lmhead_forward(m.h, m.W, m.t, m.mask, m.T)
        dh = slp.slp_lmhead_backward_accumulate(m.h, m.W, m.t, m.mask, m.T, lse, m.g, acc)
        dh_plain, _ = slp.slp_lmhead_backward(m.h, m.W, m.t, m.mask, m.T, lse, m.g)
        torch.cuda.synchronize()
        assert torch.equal(dh, dh_plain)
        t, mk = m.t.cpu().numpy(), m.mask.cpu().numpy()
        _, rlse = O.lmhead_forward(to64(m.h), to64(m.W), t, mk, m.T)
        refs.append(O.lmhead_backward(to64(m.h), to64(m.W), t, mk, m.T, rlse, to64(m.g))[1])
    grad_ok(to64(acc - acc0), refs[0] + refs[1], "accumulated dW")


def test_lmhead_matches_logits_path():
    """Fused against unfused: the LM head's logprob and lse equal those of
    slp_forward on the materialised fp32 logits h W^T, and its gradients equal
    the logits path's fp32 gradient pushed through the projection."""
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=500, V=9000, d=320, p_mask=0.7, seed=43)
    a.W = (a.W.float() * 8).to(torch.bfloat16)  # logits of a few units
    lp, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T)
    dh, dW = slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, lse, a.g)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        x = a.h.float() @ a.W.float().t()  # fp32 logits, no TF32
        lp2, lse2 = slp.slp_forward(x, a.t, a.mask, a.T)
        gx = slp.slp_backward(x, a.t, a.mask, a.T, lse2, a.g)
        dh2 = gx @ a.W.float()
        dW2 = gx.t() @ a.h.float()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    torch.cuda.synchronize()
    assert float((lp - lp2).abs().max()) <= 1e-4 and float((lse - lse2).abs().max()) <= 1e-4
    for got, ref, what in ((dh.float(), dh2, "dh"), (dW.float(), dW2, "dW")):
        cos = float((got * ref).sum() / (got.norm() * ref.norm()))
        frob = float((got - ref).norm() / ref.norm())
        assert cos >= 0.9999 and frob <= 1e-2, f"{what}: cosine {cos:.6f} frob {frob:.3e}"


def test_dirty_workspace_is_harmless():
    """Every workspace value a call reads it wrote first: the scan zeroes the
    counters from which the GEMMs' pairs claim their units (each GEMM zeroes
    the next launch's) and the forward's slab counters.  A workspace filled
    with 0xFF before a forward, the backward on the forward's leftovers, then
    a forward with another mask and temperature on a workspace filled with
    0x7F: each matches the oracle."""
    dev = device()
    N, V, d = 700, 30000, 256
    a = W.make_lmhead_inputs(device=dev, N=N, V=V, d=d, p_mask=0.6, seed=77)
    ws = torch.full((slp.slp_lmhead_workspace_size(N, V, d),), 0xFF, dtype=torch.uint8,
                    device=dev)
    lp, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T, ws=ws)
    dh, dW = slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, lse, a.g, ws=ws)
    mask2 = (torch.arange(N, device=dev) % 3 != 0).to(torch.uint8)
    ws.fill_(0x7F)
    lp2, lse2 = slp.slp_lmhead_forward(a.h, a.W, a.t, mask2, 0.6, ws=ws)
    torch.cuda.synchronize()
    h64, W64 = to64(a.h), to64(a.W)
    t, m, g = a.t.cpu().numpy(), a.mask.cpu().numpy(), to64(a.g)
    rlp, rlse = O.lmhead_forward(h64, W64, t, m, a.T)
    assert_close_nan(to64(lp), rlp, TOL_LP, "logprob")
    assert_close_nan(to64(lse), rlse, TOL_LP, "lse")
    rdh, rdW = O.lmhead_backward(h64, W64, t, m, a.T, rlse, g)
    grad_ok(to64(dh), rdh, "dh")
    grad_ok(to64(dW), rdW, "dW")
    rlp2, rlse2 = O.lmhead_forward(h64, W64, t, mask2.cpu().numpy(), 0.6)
    assert_close_nan(to64(lp2), rlp2, TOL_LP, "logprob, second mask")
    assert_close_nan(to64(lse2), rlse2, TOL_LP, "lse, second mask")


def test_two_streams_at_once():
    """Two forward + backward calls issued on two streams at once, each with
    its own workspace: the second call's CTA pairs start while the first's
    still hold SMs, and both claim their units from their own counters.  Each
    matches the oracle."""
    dev = device()
    cases = [W.make_lmhead_inputs(device=dev, N=600, V=24000, d=256, p_mask=0.7, seed=s)
             for s in (81, 82)]
    streams = [torch.cuda.Stream(device=dev) for _ in cases]
    outs = []
    torch.cuda.synchronize()
    for a, st in zip(cases, streams):
        N, V, d = a.h.shape[0], a.W.shape[0], a.h.shape[1]
        ws = torch.empty(slp.slp_lmhead_workspace_size(N, V, d), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(st):
            lp, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T, ws=ws, stream=st)
            dh, dW = slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, lse, a.g, ws=ws,
                                             stream=st)
        outs.append((lp, lse, dh, dW, ws))
    torch.cuda.synchronize()
    for a, (lp, lse, dh, dW, _) in zip(cases, outs):
        h64, W64 = to64(a.h), to64(a.W)
        t, m, g = a.t.cpu().numpy(), a.mask.cpu().numpy(), to64(a.g)
        rlp, rlse = O.lmhead_forward(h64, W64, t, m, a.T)
        assert_close_nan(to64(lp), rlp, TOL_LP, "logprob")
        rdh, rdW = O.lmhead_backward(h64, W64, t, m, a.T, rlse, g)
        grad_ok(to64(dh), rdh, "dh")
        grad_ok(to64(dW), rdW, "dW")


@pytest.mark.parametrize("extra", ["max", "middle", "default-less", "min"])
def test_backward_chunk_width_follows_the_workspace(extra):
    """The backward's vocabulary chunk follows the workspace: the whole
    vocabulary (slp_lmhead_workspace_size_max), 131072 + the rest (a little
    less), 32768 (a little less than the default 65536) and 16384 columns
    (slp_lmhead_workspace_size_min).  Each agrees with the oracle and with the
    default chunking."""
    dev = device()
    N, V, d = 200, 140000, 128
    a = W.make_lmhead_inputs(device=dev, N=N, V=V, d=d, p_mask=0.8, seed=44)
    a.W = (a.W.float() * 5).to(torch.bfloat16)
    lp, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T)
    big = slp.slp_lmhead_workspace_size_max(N, V, d)
    dflt = slp.slp_lmhead_workspace_size(N, V, d)
    small = slp.slp_lmhead_workspace_size_min(N, V, d)
    assert big > dflt > small
    nbytes = {"max": big, "middle": big - 256, "default-less": dflt - 256, "min": small}[extra]
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dh, dW = slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, lse, a.g, ws=ws)
    dh0, dW0 = slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, lse, a.g)
    torch.cuda.synchronize()
    h64, W64 = to64(a.h), to64(a.W)
    t, m, g = a.t.cpu().numpy(), a.mask.cpu().numpy(), to64(a.g)
    _, rlse = O.lmhead_forward(h64, W64, t, m, a.T)
    rdh, rdW = O.lmhead_backward(h64, W64, t, m, a.T, rlse, g)
    grad_ok(to64(dh), rdh, "dh")
    grad_ok(to64(dW), rdW, "dW")
    grad_ok(to64(dh), to64(dh0), "dh against the default chunking")
    grad_ok(to64(dW), to64(dW0), "dW against the default chunking")


def test_wait_that_runs_out_flags_the_call_and_the_stream_recovers():
    """With the wait bound set to 1 ns, the LM-head GEMMs' pipeline waits run
    out: the forward and the backward return, SLP_DEVICE_ERR_TIMEOUT is set in
    the error word, and normal calls right after, on the same stream, match
    the oracle (the kernels drained their copies and tensor-core work and
    freed their tensor memory instead of hanging)."""
    from vocab_selected_token_gb300 import _lib
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=512, V=32768, d=2560, seed=41, p_mask=0.8)
    flagged = {"forward": False, "backward": False}
    prev = slp.slp_lmhead_set_wait_limit_ns(1)
    try:
        assert prev == 2_000_000_000  # the default bound
        for _ in range(5):  # every CTA's first few waits may still be met in time
            err = torch.zeros(1, dtype=torch.int32, device=dev)
            _, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T, err=err)
            torch.cuda.synchronize()
            flagged["forward"] |= bool(int(err.item()) & _lib.SLP_DEVICE_ERR_TIMEOUT)
            err = torch.zeros(1, dtype=torch.int32, device=dev)
            slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, torch.zeros_like(lse), a.g,
                                    err=err)
            torch.cuda.synchronize()
            flagged["backward"] |= bool(int(err.item()) & _lib.SLP_DEVICE_ERR_TIMEOUT)
            if all(flagged.values()):
                break
    finally:
        assert slp.slp_lmhead_set_wait_limit_ns(0) == 1
    assert flagged["forward"] and flagged["backward"], flagged
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse, dh, dW = run_fwd_bwd(a, err=err)
    assert int(err.item()) == 0
    h64, W64 = to64(a.h), to64(a.W)
    t, m, g = a.t.cpu().numpy(), a.mask.cpu().numpy(), to64(a.g)
    rlp, rlse = O.lmhead_forward(h64, W64, t, m, a.T)
    assert_close_nan(to64(lp), rlp, TOL_LP, "logprob after the timed-out calls")
    rdh, rdW = O.lmhead_backward(h64, W64, t, m, a.T, rlse, g)
    grad_ok(to64(dh), rdh, "dh after the timed-out calls")
    grad_ok(to64(dW), rdW, "dW after the timed-out calls")
