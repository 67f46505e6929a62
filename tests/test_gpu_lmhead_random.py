"""GPU: a seeded sweep of random shapes through the fused LM head
(slp_lmhead_forward / slp_lmhead_backward): row counts that leave a ragged row
block, vocabularies from 1 column to several chunks' worth of tiles, hidden
sizes that are multiples of 64 but not of the 256-column tile, temperatures,
mask densities and logit scales.  Every output is compared with the oracle,
using the LM-head tolerances.

With V = 1 the exact gradients are zero.  The kernels recompute p from the
fp32 lse and get 1 - p of order 1e-7, so there the check is an absolute bound
instead of cosine and Frobenius (which are undefined against a zero
reference)."""

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


def _case(seed):
    r = np.random.default_rng(2000 + seed)
    N = int(r.integers(1, 700))
    V = int(r.choice([1, 7, 256, 1000, 5003, 33000]))
    d = int(r.choice([64, 128, 192, 320, 512]))
    T = float(r.choice([1.0, 0.7, 1.9]))
    pm = float(r.choice([1.0, 0.9, 0.5, 0.1]))
    scale = float(r.choice([1.0, 5.0, 20.0]))
    return N, V, d, T, pm, scale


def _grad_check(got, ref, what):
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    nr = np.linalg.norm(ref)
    if nr == 0:
        assert np.abs(got).max(initial=0.0) <= 1e-4, f"{what}: zero reference, got {np.abs(got).max()}"
        return
    cos = float(got @ ref / (np.linalg.norm(got) * nr + 1e-300))
    frob = float(np.linalg.norm(got - ref) / nr)
    assert cos >= COS_MIN and frob <= FROB_MAX, f"{what}: cosine {cos:.6f} frob {frob:.3e}"


EDGES = [
    # N, V, d, T, p_mask, scale
    (130, 1, 128, 1.0, 0.5, 5.0),       # one vocabulary column: zero gradients
    (700, 1, 64, 0.7, 1.0, 20.0),
    (1, 33000, 2560, 1.0, 1.0, 5.0),    # a single row, the workload's hidden size
    (129, 257, 64, 1.3, 1.0, 20.0),     # one row and one column past a tile
    (70, 70001, 64, 1.0, 0.5, 5.0),     # two backward vocabulary chunks, the second ragged
    (300, 140000, 128, 0.8, 0.9, 1.0),  # three chunks
]


@pytest.mark.parametrize("seed", range(16))
def test_random_lmhead(seed):
    _run(*_case(seed), seed=300 + seed)


@pytest.mark.parametrize("case", EDGES, ids=lambda v: str(v))
def test_lmhead_edges(case):
    _run(*case, seed=400 + EDGES.index(case))


def _run(N, V, d, T, pm, scale, seed, err=None):
    dev = device()
    a = W.make_lmhead_inputs(device=dev, N=N, V=V, d=d, p_mask=pm, seed=seed)
    a.W = (a.W.float() * scale).to(torch.bfloat16)
    a.T = T
    lp, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, T, err=err)
    dh, dW = slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, T, lse, a.g, err=err)
    torch.cuda.synchronize()
    h64, W64 = to64(a.h), to64(a.W)
    t, m, g = a.t.cpu().numpy(), a.mask.cpu().numpy(), to64(a.g)
    rlp, rlse = O.lmhead_forward(h64, W64, t, m, T)
    assert_close_nan(to64(lp), rlp, TOL_LP, "logprob")
    assert_close_nan(to64(lse), rlse, TOL_LP, "lse")
    rdh, rdW = O.lmhead_backward(h64, W64, t, m, T, rlse, g)
    _grad_check(to64(dh), rdh, "dh")
    _grad_check(to64(dW), rdW, "dW")
    off = torch.as_tensor(m == 0, device=dev)
    assert bool((dh[off].view(torch.int16) == 0).all()), "masked dh rows not +0.0"
    assert bool((lp[off] == 0).all()) and bool((lse[off] == 0).all())
