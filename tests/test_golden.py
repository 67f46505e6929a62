"""CPU-only: stored oracle cases against their closed forms, and the oracle
against what it stored (regression)."""

import json
import math
import os

import numpy as np
import pytest

from oracle import slp_oracle as O

CASES = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "oracle_cases.json")))["cases"]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["name"])
def test_golden_closed_form(case):
    lp = np.array(case["logprob"])
    ref = np.array(case["closed_form_lp"])
    assert np.allclose(lp, ref, rtol=0, atol=case["closed_form_tol"])
    gx = np.array(case["grad_x"])
    # each gradient row sums to zero and the target entry is g (1 - p_t) / T
    assert np.allclose(gx.sum(axis=1), 0.0, atol=1e-14)
    g = np.array(case["g"])
    T = case["T"]
    for n, t in enumerate(case["t"]):
        assert math.isclose(gx[n, t], g[n] * (1 - math.exp(ref[n])) / T,
                            rel_tol=0, abs_tol=max(case["closed_form_tol"], 1e-15) * 4)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["name"])
def test_oracle_reproduces_golden(case):
    x = np.array(case["x"])
    lp, lse = O.selected_logprob_forward(x, case["t"], None, case["T"])
    gx = O.selected_logprob_backward(x, case["t"], None, case["T"], lse, case["g"])
    assert np.array_equal(lp, np.array(case["logprob"]))
    assert np.array_equal(lse, np.array(case["lse"]))
    assert np.array_equal(gx, np.array(case["grad_x"]))
