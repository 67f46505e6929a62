"""CPU-only: the oracle against its pins, and planted mistakes against the pins."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import slp_oracle as O
from tests.oracle_pins import ALL_PINS, Impl, run_all

ORACLE = Impl(O.selected_logprob_forward, O.selected_logprob_backward,
              O.lmhead_forward, O.lmhead_backward)


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(ORACLE)


# --- planted mistakes (all in copies of the oracle, on the CPU) --------------

def _fwd_raw_target(x, t, mask, T):
    lp, lse = O.selected_logprob_forward(x, t, mask, T)
    x = np.asarray(x, np.float64)
    z_t = x[np.arange(x.shape[0]), np.asarray(t)] / T
    return lp - z_t + z_t * T, lse          # target logit not divided by T


def _fwd_off_by_one(x, t, mask, T):
    V = np.asarray(x).shape[1]
    return O.selected_logprob_forward(x, (np.asarray(t) + 1) % V, mask, T)


def _fwd_no_max(x, t, mask, T):
    x = np.asarray(x, np.float64)
    N = x.shape[0]
    with np.errstate(all="ignore"):
        lse = np.log(np.sum(np.exp(x / T), axis=1))
        lp = x[np.arange(N), np.asarray(t)] / T - lse
    if mask is not None:
        m = np.asarray(mask) != 0
        lp, lse = np.where(m, lp, 0.0), np.where(m, lse, 0.0)
    return lp, lse


def _bwd_sign(x, t, mask, T, lse, g):
    return -O.selected_logprob_backward(x, t, mask, T, lse, g)


def _bwd_no_T(x, t, mask, T, lse, g):
    return O.selected_logprob_backward(x, t, mask, T, lse, g) * T


def _bwd_no_onehot(x, t, mask, T, lse, g):
    gx = O.selected_logprob_backward(x, t, mask, T, lse, g)
    N = gx.shape[0]
    active = np.ones(N, bool) if mask is None else np.asarray(mask) != 0
    gx[np.arange(N), np.asarray(t)] -= np.where(active, np.asarray(g, np.float64) / T, 0.0)
    return gx


def _bwd_ignores_mask(x, t, mask, T, lse, g):
    _, lse_all = O.selected_logprob_forward(x, t, None, T)
    return O.selected_logprob_backward(x, t, None, T, lse_all, g)


def _lmh_bwd_wrong_rows(h, W, t, mask, T, lse, g):
    dh, dW = O.lmhead_backward(h, W, t, mask, T, lse, g)
    h = np.asarray(h, np.float64)
    rows = np.nonzero(np.asarray(mask) != 0)[0]
    # pair each dz row with the wrong hidden row (reversed order)
    x = O.lmhead_logits(h[rows], W)
    dz = O.selected_logprob_backward(x, np.asarray(t)[rows], None, T,
                                     np.asarray(lse)[rows], np.asarray(g)[rows])
    return dh, dz.T @ h[rows[::-1]]


def _lmh_fwd_no_T(h, W, t, mask, T):
    return O.lmhead_forward(h, W, t, mask, 1.0)


MUTANTS = {
    "fwd_raw_target": Impl(_fwd_raw_target, O.selected_logprob_backward, O.lmhead_forward, O.lmhead_backward),
    "fwd_off_by_one": Impl(_fwd_off_by_one, O.selected_logprob_backward, O.lmhead_forward, O.lmhead_backward),
    "fwd_no_max": Impl(_fwd_no_max, O.selected_logprob_backward, O.lmhead_forward, O.lmhead_backward),
    "bwd_sign": Impl(O.selected_logprob_forward, _bwd_sign, O.lmhead_forward, O.lmhead_backward),
    "bwd_no_T": Impl(O.selected_logprob_forward, _bwd_no_T, O.lmhead_forward, O.lmhead_backward),
    "bwd_no_onehot": Impl(O.selected_logprob_forward, _bwd_no_onehot, O.lmhead_forward, O.lmhead_backward),
    "bwd_ignores_mask": Impl(O.selected_logprob_forward, _bwd_ignores_mask, O.lmhead_forward, O.lmhead_backward),
    "lmhead_bwd_wrong_rows": Impl(O.selected_logprob_forward, O.selected_logprob_backward, O.lmhead_forward, _lmh_bwd_wrong_rows),
    "lmhead_fwd_no_T": Impl(O.selected_logprob_forward, O.selected_logprob_backward, _lmh_fwd_no_T, O.lmhead_backward),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    with pytest.raises(AssertionError):
        run_all(MUTANTS[name])


# --- bfloat16 decoding -------------------------------------------------------

def test_decode_bf16_known_patterns():
    pats = np.array([0x3F80, 0xC000, 0x7F80, 0xFF80, 0x0001, 0x4049, 0x0000, 0x8000], np.uint16)
    val = O.decode_bf16(pats)
    assert val[0] == 1.0 and val[1] == -2.0
    assert val[2] == np.inf and val[3] == -np.inf
    assert val[4] == 2.0 ** -133
    assert val[5] == 3.140625
    assert val[6] == 0.0 and val[7] == 0.0 and np.signbit(val[7])


def test_decode_bf16_all_patterns_match_torch():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.decode_bf16(pats)
    theirs = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).double().numpy()
    same = (ours == theirs) | (np.isnan(ours) & np.isnan(theirs))
    assert same.all()


def test_sampled_lmhead_gradients_match_full_backward():
    """The one-row-at-a-time dh / dW helpers equal the finite-difference-pinned
    full backward."""
    r = np.random.default_rng(12)
    N, d, V, T = 9, 8, 30, 0.8
    h = r.normal(0, 1, (N, d))
    W = r.normal(0, 0.4, (V, d))
    t = r.integers(0, V, N)
    g = r.uniform(-1, 1, N)
    mask = (r.random(N) < 0.6).astype(np.uint8)
    _, lse = O.lmhead_forward(h, W, t, mask, T)
    dh, dW = O.lmhead_backward(h, W, t, mask, T, lse, g)
    rows = [0, 3, 8, 5]
    assert np.allclose(O.lmhead_dh_rows(h, W, t, mask, T, lse, g, rows), dh[rows], rtol=1e-12, atol=1e-14)
    vr = [0, 7, 29, 13]
    assert np.allclose(O.lmhead_dW_rows(h, W, t, mask, T, lse, g, vr), dW[vr], rtol=1e-12, atol=1e-14)


def test_entropy_pins():
    from tests.oracle_pins import pin_entropy_closed_forms, pin_entropy_finite_differences
    pin_entropy_closed_forms(O.entropy_forward)
    pin_entropy_finite_differences(O.entropy_forward, O.entropy_backward)


def test_entropy_pins_catch_planted_mistakes():
    from tests.oracle_pins import pin_entropy_closed_forms, pin_entropy_finite_differences

    def fwd_no_T(x, t, mask, T):
        return O.entropy_forward(np.asarray(x, np.float64) * T, t, mask, T)

    def bwd_wrong_sign(x, t, mask, T, lse, H, g, gH):
        return O.entropy_backward(x, t, mask, T, lse, H, g, -np.asarray(gH))

    def bwd_no_H(x, t, mask, T, lse, H, g, gH):
        return O.entropy_backward(x, t, mask, T, lse, np.zeros_like(np.asarray(H)), g, gH)

    with pytest.raises(AssertionError):
        pin_entropy_closed_forms(fwd_no_T)
    for bad in (bwd_wrong_sign, bwd_no_H):
        with pytest.raises(AssertionError):
            pin_entropy_finite_differences(O.entropy_forward, bad)


def test_topk_kl_pins():
    from tests.oracle_pins import (pin_topk_kl_clamp, pin_topk_kl_finite_differences,
                                   pin_topk_kl_library)
    pin_topk_kl_library(O.topk_kl_forward)
    pin_topk_kl_clamp(O.topk_kl_forward)
    pin_topk_kl_finite_differences(O.topk_kl_forward, O.topk_kl_backward)


def test_topk_kl_pins_catch_planted_mistakes():
    from tests.oracle_pins import pin_topk_kl_finite_differences, pin_topk_kl_library

    def fwd_unnormalised(x, ids, lt, mask, T, clamp):   # forgets the student's lse
        kl, sm, tm, lse = O.topk_kl_forward(x, ids, lt, mask, T, clamp)
        return kl + np.asarray(np.exp(lt)).sum(axis=1) * lse, sm, tm, lse

    def bwd_no_dense(x, ids, lt, mask, T, clamp, lse, g):  # drops the P q term
        gx = O.topk_kl_backward(x, ids, lt, mask, T, clamp, lse, g)
        q = np.exp(np.asarray(x) / T - np.asarray(lse)[:, None])
        return gx - 0.5 * np.asarray(g)[:, None] * q / T

    def bwd_ignores_clamp(x, ids, lt, mask, T, clamp, lse, g):
        return O.topk_kl_backward(x, ids, lt, mask, T, None, lse, g)

    with pytest.raises(AssertionError):
        pin_topk_kl_library(fwd_unnormalised)
    for bad in (bwd_no_dense, bwd_ignores_clamp):
        with pytest.raises(AssertionError):
            pin_topk_kl_finite_differences(O.topk_kl_forward, bad)
