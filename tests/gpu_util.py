"""Shared helpers of the GPU parity tests: build the library once, compare the
CUDA outputs of chosen rows with the CPU oracle at the stated tolerances."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import slp_oracle as O

# Tolerances of the logits-input path (fp32 logprob absolute; per-element
# gradient bound 2^-8 |ref| + 1e-6, i.e. bf16 rounding plus fp32 noise).
TOL_LP = 2e-5
GRAD_REL = 2.0 ** -8
GRAD_ABS = 1e-6


def device():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from vocab_selected_token_gb300 import build
    build.build()
    return torch.device("cuda:0")


def to64(x: torch.Tensor) -> np.ndarray:
    return x.detach().double().cpu().numpy()


def assert_close_nan(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    same_nan = np.isnan(a) == np.isnan(b)
    assert same_nan.all(), f"{what}: NaN pattern differs at {np.flatnonzero(~same_nan)[:5]}"
    same_inf = (np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))) | ~(np.isinf(a) | np.isinf(b))
    assert same_inf.all(), f"{what}: inf pattern differs"
    fin = np.isfinite(a) & np.isfinite(b)
    if fin.any():
        err = np.abs(a[fin] - b[fin]).max()
        assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


def assert_grad_close(gx, ref, what="grad", floor=None):
    """Per element |gx - ref| <= 2^-8 |ref| + 1e-6 (+ floor[row] when given)."""
    gx = np.asarray(gx, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = GRAD_REL * np.abs(ref) + GRAD_ABS
    if floor is not None:
        bound = bound + np.asarray(floor, np.float64).reshape(-1, 1)
    bad = np.abs(gx - ref) > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements outside 2^-8|ref|+1e-6, first at "
                             f"{tuple(i)}: got {gx[tuple(i)]!r} ref {ref[tuple(i)]!r}")


def lse_floor(x64, rlse, g, T):
    """Absolute error floor of a gradient recomputed from an fp32 lse: the
    exponent x/T - lse carries about ulp(|x/T|) + ulp(|lse|), so every element
    (the target's 1 - p above all) can be off by |g/T| times that."""
    big = np.maximum(np.abs(np.nan_to_num(x64, neginf=0.0)).max(axis=1) / T, np.abs(rlse))
    return np.abs(g) / T * 4.0 * big * 2.0 ** -24


def check_rows(x, t, mask, T, g, lp, lse, gx, rows, fp32_floor=False):
    """Compare rows `rows` of the CUDA outputs with the oracle run on the same
    rows of the same inputs.  fp32_floor adds lse_floor to the gradient bound
    (for inputs far outside the workloads' range, see lse_floor)."""
    rows = np.asarray(sorted(set(int(r) for r in rows)))
    ridx = torch.as_tensor(rows, device=x.device)
    x64 = to64(x[ridx])
    tr = t[ridx].cpu().numpy()
    mr = None if mask is None else mask[ridx].cpu().numpy()
    gr = to64(g[ridx])
    rlp, rlse = O.selected_logprob_forward(x64, tr, mr, T)
    assert_close_nan(to64(lp[ridx]), rlp, TOL_LP, "logprob")
    assert_close_nan(to64(lse[ridx]), rlse, TOL_LP, "lse")
    if gx is not None:
        rgx = O.selected_logprob_backward(x64, tr, mr, T, rlse, gr)
        floor = lse_floor(x64, rlse, gr, T) if fp32_floor else None
        assert_grad_close(to64(gx[ridx]), rgx, floor=floor)
        if mr is not None:
            off = mr == 0
            if off.any():
                z = gx[ridx][torch.as_tensor(off, device=x.device)].contiguous()
                bits = z.view(torch.int32) if z.dtype == torch.float32 else z.view(torch.int16)
                assert bool((bits == 0).all()), "masked gradient rows not +0.0"
