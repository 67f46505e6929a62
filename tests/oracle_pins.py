"""Pins that tie the CPU oracle to facts other than itself.

Each pin takes an implementation bundle (forward, backward, lmhead_forward,
lmhead_backward with the oracle's signatures) and raises AssertionError when
the bundle disagrees with a closed form, an invariant, finite differences or
an independent library routine.  ``tests/test_oracle_pins.py`` runs every pin
on the oracle (all must pass) and on planted-mistake variants of it (each must
be caught by at least one pin).
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable

import numpy as np
import torch
import torch.nn.functional as F


@dataclass
class Impl:
    forward: Callable
    backward: Callable
    lmhead_forward: Callable
    lmhead_backward: Callable


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol, atol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    ok = np.isclose(a, b, rtol=rtol, atol=atol, equal_nan=True)
    assert ok.all(), f"{what}: max |diff| {np.nanmax(np.abs(a - b))}"


# --- forward -----------------------------------------------------------------

def pin_cross_entropy_identity(impl: Impl):
    """logprob == -cross_entropy(x/T, t) at label smoothing 0 (Megatron-LM
    issue #6700, "Proposed solution"), checked against torch's fp64 CPU
    cross_entropy and logsumexp, which the oracle does not call."""
    r = _rng(1)
    for (N, V, T) in [(16, 37, 0.7), (5, 2, 1.0), (9, 1000, 1.3)]:
        x = r.normal(0, 3, (N, V))
        t = r.integers(0, V, N)
        lp, lse = impl.forward(x, t, None, T)
        xt = torch.from_numpy(x / T)
        ce = F.cross_entropy(xt, torch.from_numpy(t), reduction="none").numpy()
        _close(lp, -ce, 1e-12, 1e-12, "lp vs -cross_entropy")
        _close(lse, torch.logsumexp(xt, dim=1).numpy(), 1e-12, 1e-12, "lse vs logsumexp")


def pin_normalisation(impl: Impl):
    """sum over all targets v of exp(logprob(v)) is 1 for every row."""
    r = _rng(2)
    N, V, T = 4, 50, 0.9
    x = r.normal(0, 2, (N, V))
    tot = np.zeros(N)
    for v in range(V):
        lp, _ = impl.forward(x, np.full(N, v), None, T)
        tot += np.exp(lp)
    _close(tot, np.ones(N), 1e-12, 0, "sum_v exp(lp)")


def pin_shift_invariance(impl: Impl):
    """lp(x + c_n) == lp(x) and lse(x + c_n) == lse(x) + c_n / T per row."""
    r = _rng(3)
    N, V, T = 6, 77, 0.6
    x = r.normal(0, 2, (N, V))
    c = r.normal(0, 50, N)
    t = r.integers(0, V, N)
    lp0, lse0 = impl.forward(x, t, None, T)
    lp1, lse1 = impl.forward(x + c[:, None], t, None, T)
    _close(lp1, lp0, 1e-11, 1e-11, "shifted lp")
    _close(lse1, lse0 + c / T, 1e-11, 1e-11, "shifted lse")


def pin_uniform(impl: Impl):
    """Constant logits: lp = -log V and grad = g (1[v=t] - 1/V) / T."""
    for V in (1, 2, 7, 151936):
        N, T = 3, 0.7
        x = np.full((N, V), 2.5)
        t = np.array([0, V - 1, V // 2])
        g = np.array([1.0, -0.5, 0.25])
        lp, lse = impl.forward(x, t, None, T)
        _close(lp, np.full(N, -math.log(V)), 1e-13, 1e-13, f"uniform lp V={V}")
        _close(lse, np.full(N, 2.5 / T + math.log(V)), 1e-13, 1e-13, "uniform lse")
        if V <= 7:
            gx = impl.backward(x, t, None, T, lse, g)
            ref = -np.outer(g, np.full(V, 1.0 / V)) / T
            ref[np.arange(N), t] += g / T
            _close(gx, ref, 1e-13, 1e-15, f"uniform grad V={V}")


def pin_two_class(impl: Impl):
    """V = 2: lp = -log(1 + exp((x_other - x_target)/T)) (log-sigmoid)."""
    r = _rng(4)
    N, T = 32, 1.7
    x = r.normal(0, 5, (N, 2))
    t = r.integers(0, 2, N)
    lp, _ = impl.forward(x, t, None, T)
    ref = np.array([-math.log1p(math.exp((x[n, 1 - t[n]] - x[n, t[n]]) / T)) for n in range(N)])
    _close(lp, ref, 1e-12, 1e-13, "log-sigmoid")


def pin_spike(impl: Impl):
    """Zeros with one spike a at column j: lp(t=j) = a/T - log(e^{a/T} + V - 1),
    lp(t!=j) = -log(e^{a/T} + V - 1)."""
    V, T, a, j = 1000, 0.8, 8.0, 123
    x = np.zeros((2, V))
    x[:, j] = a
    t = np.array([j, 7])
    lp, _ = impl.forward(x, t, None, T)
    den = math.log(math.exp(a / T) + V - 1)
    _close(lp, [a / T - den, -den], 1e-13, 1e-13, "spike")


def pin_extremes(impl: Impl):
    """Large magnitudes and -inf entries stay finite and match torch's fp64
    log_softmax; an all -inf row is NaN; a target on a -inf column is -inf."""
    r = _rng(5)
    N, V, T = 5, 300, 1.0
    x = r.normal(0, 4, (N, V))
    x[r.random((N, V)) < 0.05] = 1000.0
    x[r.random((N, V)) < 0.05] = -1000.0
    x[1, 10:40] = -np.inf
    t = r.integers(0, V, N)
    t[1] = 50
    lp, lse = impl.forward(x, t, None, T)
    ref = torch.log_softmax(torch.from_numpy(x), dim=1).numpy()[np.arange(N), t]
    assert np.isfinite(lp).all() and np.isfinite(lse).all(), "extreme logits not finite"
    _close(lp, ref, 1e-12, 1e-10, "extreme lp")
    y = np.full((1, 4), -np.inf)
    lpn, lsen = impl.forward(y, np.array([0]), None, 1.0)
    assert np.isnan(lpn[0]) and np.isnan(lsen[0]), "all -inf row must be NaN"
    z = np.array([[0.0, -np.inf, 1.0]])
    lpi, _ = impl.forward(z, np.array([1]), None, 1.0)
    assert lpi[0] == -np.inf, "target on a -inf column must be -inf"


# --- backward ----------------------------------------------------------------

def pin_row_sum(impl: Impl):
    """Each gradient row sums to zero (softmax sums to one)."""
    r = _rng(6)
    N, V, T = 8, 500, 0.7
    x = r.normal(0, 3, (N, V))
    t = r.integers(0, V, N)
    g = r.uniform(-1, 1, N)
    _, lse = impl.forward(x, t, None, T)
    gx = impl.backward(x, t, None, T, lse, g)
    _close(gx.sum(axis=1), np.zeros(N), 0, 1e-13, "grad row sum")


def pin_finite_differences(impl: Impl):
    """Analytic gradient of L = sum_n g_n lp_n matches central differences
    (step 1e-6) on a tiny fp64 problem."""
    r = _rng(7)
    N, V, T, hstep = 4, 9, 0.8, 1e-6
    x = r.normal(0, 1.5, (N, V))
    t = r.integers(0, V, N)
    g = r.uniform(-1, 1, N)
    _, lse = impl.forward(x, t, None, T)
    gx = impl.backward(x, t, None, T, lse, g)
    fd = np.zeros_like(x)
    for n in range(N):
        for v in range(V):
            xp = x.copy(); xp[n, v] += hstep
            xm = x.copy(); xm[n, v] -= hstep
            fd[n, v] = (np.dot(g, impl.forward(xp, t, None, T)[0]) -
                        np.dot(g, impl.forward(xm, t, None, T)[0])) / (2 * hstep)
    _close(gx, fd, 1e-7, 1e-9, "finite differences")


def pin_autograd(impl: Impl):
    """Gradient equals torch autograd through log_softmax(x/T).gather(t) in
    fp64 (the unchunked reference the NeMo-RL PR #4222 tests compare to)."""
    r = _rng(8)
    N, V, T = 6, 211, 0.65
    x = r.normal(0, 3, (N, V))
    t = r.integers(0, V, N)
    g = r.uniform(-1, 1, N)
    _, lse = impl.forward(x, t, None, T)
    gx = impl.backward(x, t, None, T, lse, g)
    xt = torch.from_numpy(x).requires_grad_(True)
    lp = torch.log_softmax(xt / T, dim=1).gather(1, torch.from_numpy(t)[:, None])[:, 0]
    (lp * torch.from_numpy(g)).sum().backward()
    _close(gx, xt.grad.numpy(), 1e-12, 1e-14, "autograd grad")


def pin_mask(impl: Impl):
    """Masked rows are exactly 0 (lp, lse and gradient); an all-one mask is the
    unmasked result; an all-zero mask gives all zeros."""
    r = _rng(9)
    N, V, T = 10, 64, 0.9
    x = r.normal(0, 2, (N, V))
    t = r.integers(0, V, N)
    g = r.uniform(-1, 1, N)
    mask = (r.random(N) < 0.5).astype(np.uint8)
    mask[0], mask[1] = 1, 0
    lp, lse = impl.forward(x, t, mask, T)
    lpu, lseu = impl.forward(x, t, None, T)
    off = mask == 0
    assert (lp[off] == 0).all() and (lse[off] == 0).all(), "masked lp/lse not zero"
    _close(lp[~off], lpu[~off], 0, 0, "masked vs unmasked lp")
    gx = impl.backward(x, t, mask, T, lse, g)
    assert (gx[off] == 0).all(), "masked gradient rows not zero"
    gxu = impl.backward(x, t, None, T, lseu, g)
    _close(gx[~off], gxu[~off], 0, 0, "masked vs unmasked grad")
    lp1, _ = impl.forward(x, t, np.ones(N, np.uint8), T)
    _close(lp1, lpu, 0, 0, "all-one mask")
    lp0, lse0 = impl.forward(x, t, np.zeros(N, np.uint8), T)
    assert (lp0 == 0).all() and (lse0 == 0).all(), "all-zero mask"


# --- LM head -----------------------------------------------------------------

def pin_lmhead_library(impl: Impl):
    """Fused LM-head log-probs equal torch's fp64 -cross_entropy of h W^T / T on
    the active rows, zeros elsewhere."""
    r = _rng(10)
    N, d, V, T = 12, 16, 40, 0.75
    h = r.normal(0, 1, (N, d))
    W = r.normal(0, 0.3, (V, d))
    t = r.integers(0, V, N)
    mask = (r.random(N) < 0.6).astype(np.uint8)
    lp, lse = impl.lmhead_forward(h, W, t, mask, T)
    logits = torch.from_numpy(h) @ torch.from_numpy(W).T / T
    ce = F.cross_entropy(logits, torch.from_numpy(t), reduction="none").numpy()
    ref = np.where(mask != 0, -ce, 0.0)
    _close(lp, ref, 1e-12, 1e-12, "lmhead lp")
    assert (lse[mask == 0] == 0).all()


def pin_lmhead_finite_differences(impl: Impl):
    """dh and dW match central differences of L = sum_n g_n lp_n (tiny fp64)."""
    r = _rng(11)
    N, d, V, T, hs = 5, 4, 6, 0.9, 1e-6
    h = r.normal(0, 1, (N, d))
    W = r.normal(0, 0.5, (V, d))
    t = r.integers(0, V, N)
    g = r.uniform(-1, 1, N)
    mask = np.array([1, 0, 1, 1, 0], np.uint8)
    _, lse = impl.lmhead_forward(h, W, t, mask, T)
    dh, dW = impl.lmhead_backward(h, W, t, mask, T, lse, g)

    def L(hh, WW):
        return float(np.dot(g, impl.lmhead_forward(hh, WW, t, mask, T)[0]))

    fdh = np.zeros_like(h)
    for i in range(N):
        for k in range(d):
            hp = h.copy(); hp[i, k] += hs
            hm = h.copy(); hm[i, k] -= hs
            fdh[i, k] = (L(hp, W) - L(hm, W)) / (2 * hs)
    fdW = np.zeros_like(W)
    for v in range(V):
        for k in range(d):
            Wp = W.copy(); Wp[v, k] += hs
            Wm = W.copy(); Wm[v, k] -= hs
            fdW[v, k] = (L(h, Wp) - L(h, Wm)) / (2 * hs)
    _close(dh, fdh, 1e-7, 1e-9, "lmhead dh finite differences")
    _close(dW, fdW, 1e-7, 1e-9, "lmhead dW finite differences")
    assert (dh[mask == 0] == 0).all(), "masked dh rows not zero"


ALL_PINS = [
    pin_cross_entropy_identity, pin_normalisation, pin_shift_invariance,
    pin_uniform, pin_two_class, pin_spike, pin_extremes, pin_row_sum,
    pin_finite_differences, pin_autograd, pin_mask, pin_lmhead_library,
    pin_lmhead_finite_differences,
]


def run_all(impl: Impl):
    for p in ALL_PINS:
        p(impl)


# --- entropy (per-token entropy of the same softmax) ---------------------------

def pin_entropy_closed_forms(ent_fwd):
    """Uniform logits give log V; two classes give the binary entropy; a huge
    spike gives ~0; all match torch's Categorical entropy."""
    for V in (1, 3, 1000):
        x = np.full((2, V), -1.5)
        _, _, H = ent_fwd(x, np.zeros(2, int), None, 0.9)
        _close(H, np.full(2, math.log(V)), 1e-13, 1e-13, f"uniform entropy V={V}")
    r = _rng(13)
    x = r.normal(0, 2, (16, 2))
    T = 0.8
    _, _, H = ent_fwd(x, np.zeros(16, int), None, T)
    p = 1.0 / (1.0 + np.exp(-(x[:, 0] - x[:, 1]) / T))
    ref = -(p * np.log(p) + (1 - p) * np.log(1 - p))
    _close(H, ref, 1e-12, 1e-13, "binary entropy")
    x = np.zeros((1, 50)); x[0, 7] = 500.0
    _, _, H = ent_fwd(x, np.array([7]), None, 1.0)
    assert 0 <= H[0] < 1e-100 or H[0] == 0.0
    x = r.normal(0, 3, (10, 333))
    _, _, H = ent_fwd(x, r.integers(0, 333, 10), None, 1.3)
    ref = torch.distributions.Categorical(logits=torch.from_numpy(x / 1.3)).entropy().numpy()
    _close(H, ref, 1e-12, 1e-12, "Categorical entropy")


def pin_entropy_finite_differences(ent_fwd, ent_bwd):
    """Analytic gradient of sum_n (g_n lp_n + gH_n H_n) matches central
    differences; masked rows are exactly 0."""
    r = _rng(14)
    N, V, T, hs = 4, 9, 0.7, 1e-6
    x = r.normal(0, 1.5, (N, V))
    t = r.integers(0, V, N)
    g = r.uniform(-1, 1, N)
    gH = r.uniform(-1, 1, N)
    mask = np.array([1, 1, 0, 1], np.uint8)
    _, lse, H = ent_fwd(x, t, mask, T)
    gx = ent_bwd(x, t, mask, T, lse, H, g, gH)

    def L(xx):
        lp, _, HH = ent_fwd(xx, t, mask, T)
        return float(np.dot(g, lp) + np.dot(gH, HH))

    fd = np.zeros_like(x)
    for n in range(N):
        for v in range(V):
            xp = x.copy(); xp[n, v] += hs
            xm = x.copy(); xm[n, v] -= hs
            fd[n, v] = (L(xp) - L(xm)) / (2 * hs)
    _close(gx, fd, 1e-7, 1e-9, "entropy finite differences")
    assert (gx[2] == 0).all()


# --- top-k forward KL ------------------------------------------------------------

def pin_topk_kl_library(kl_fwd):
    """kl equals torch's kl_div with log targets over the support; a teacher
    equal to the student on the whole vocabulary gives kl = 0 and both masses 1."""
    r = _rng(15)
    N, V, K, T = 6, 200, 16, 0.8
    x = r.normal(0, 2, (N, V))
    ids = np.stack([r.choice(V, K, replace=False) for _ in range(N)])
    lt = np.log(r.dirichlet(np.ones(K), N) * 0.9)
    kl, sm, tm, lse = kl_fwd(x, ids, lt, None, T, None)
    ls = x[np.arange(N)[:, None], ids] / T - lse[:, None]
    ref = [float(F.kl_div(torch.from_numpy(ls[n]), torch.from_numpy(lt[n]), log_target=True,
                          reduction="sum")) for n in range(N)]
    _close(kl, ref, 1e-12, 1e-13, "top-k kl vs kl_div")
    _close(tm, np.full(N, 0.9), 1e-12, 0, "teacher mass")
    _close(sm, np.exp(ls).sum(axis=1), 1e-12, 0, "student mass")
    full = np.tile(np.arange(V), (N, 1))
    lt_s = x / T - torch.logsumexp(torch.from_numpy(x / T), dim=1).numpy()[:, None]
    kl0, sm0, tm0, _ = kl_fwd(x, full, lt_s, None, T, None)
    _close(kl0, np.zeros(N), 0, 1e-12, "self kl")
    _close(sm0, np.ones(N), 1e-12, 0, "full student mass")


def pin_topk_kl_clamp(kl_fwd):
    """With a clamp, terms below it use the clamp value."""
    x = np.array([[0.0, -30.0, 1.0, 2.0]])
    ids = np.array([[1, 2]])
    lt = np.log(np.array([[0.5, 0.25]]))
    kl, _, _, lse = kl_fwd(x, ids, lt, None, 1.0, -10.0)
    ls2 = 1.0 - lse[0]
    ref = 0.5 * (np.log(0.5) + 10.0) + 0.25 * (np.log(0.25) - ls2)
    _close(kl, [ref], 1e-13, 1e-13, "clamped kl")


def pin_topk_kl_finite_differences(kl_fwd, kl_bwd):
    r = _rng(16)
    N, V, K, T, hs = 3, 11, 4, 0.9, 1e-6
    x = r.normal(0, 1.5, (N, V))
    x[1, 3] = -25.0          # far below the clamp: flat side
    ids = np.array([[0, 5, 5, 9], [3, 1, 2, 10], [4, 6, 7, 8]])   # a repeated id too
    lt = np.log(r.dirichlet(np.ones(K), N) * 0.8)
    g = r.uniform(-1, 1, N)
    mask = np.array([1, 1, 0], np.uint8)
    for clamp in (None, -10.0):
        kl, _, _, lse = kl_fwd(x, ids, lt, mask, T, clamp)
        gx = kl_bwd(x, ids, lt, mask, T, clamp, lse, g)

        def L(xx):
            return float(np.dot(g, kl_fwd(xx, ids, lt, mask, T, clamp)[0]))

        fd = np.zeros_like(x)
        for n in range(N):
            for v in range(V):
                xp = x.copy(); xp[n, v] += hs
                xm = x.copy(); xm[n, v] -= hs
                fd[n, v] = (L(xp) - L(xm)) / (2 * hs)
        _close(gx, fd, 1e-6, 1e-9, f"top-k kl finite differences clamp={clamp}")
        assert (gx[2] == 0).all()
