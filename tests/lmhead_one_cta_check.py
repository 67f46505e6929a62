"""Run in a child process by tests/test_gpu_lmhead_one_cta.py, with
SLP_LMHEAD_CTA_PAIRS=0 in its environment: the LM-head calls in their
one-CTA form (128 x 256 tiles, one CTA per SM), against the fp64 oracle,
including a wait bound short enough to run out.  Prints the default
workspace size for the lmhead workload's sizes (it differs between the two
forms) and exits non-zero on any mismatch."""

from __future__ import annotations

import sys

import numpy as np
import torch

import vocab_selected_token_gb300 as slp
from oracle import slp_oracle as O
from tests.gpu_util import assert_close_nan, device, to64
from vocab_selected_token_gb300 import _lib
from vocab_selected_token_gb300 import workloads as W


def grad_ok(got, ref, what):
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    cos = float(got @ ref / (np.linalg.norm(got) * np.linalg.norm(ref) + 1e-300))
    frob = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert cos >= 0.999 and frob <= 1e-2, f"{what}: cosine {cos:.6f} frob {frob:.3e}"


def check(a, lp, lse, dh, dW):
    h64, W64 = to64(a.h), to64(a.W)
    t, m, g = a.t.cpu().numpy(), a.mask.cpu().numpy(), to64(a.g)
    rlp, rlse = O.lmhead_forward(h64, W64, t, m, a.T)
    assert_close_nan(to64(lp), rlp, 5e-3, "logprob")
    rdh, rdW = O.lmhead_backward(h64, W64, t, m, a.T, rlse, g)
    grad_ok(to64(dh), rdh, "dh")
    grad_ok(to64(dW), rdW, "dW")


def main() -> int:
    dev = device()
    print("workspace", slp.slp_lmhead_workspace_size(8192, 151936, 2560), flush=True)
    for N, V, d, pm in ((300, 1000, 128, 0.5), (130, 4096, 2560, 0.9), (700, 9000, 256, 0.7)):
        a = W.make_lmhead_inputs(device=dev, N=N, V=V, d=d, p_mask=pm, seed=17)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        lp, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T, err=err)
        dh, dW = slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, lse, a.g, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        check(a, lp, lse, dh, dW)
    # a wait bound of 1 ns: both calls flag the timeout; normal calls after them match
    a = W.make_lmhead_inputs(device=dev, N=512, V=32768, d=2560, seed=41, p_mask=0.8)
    slp.slp_lmhead_set_wait_limit_ns(1)
    flagged = [False, False]
    try:
        for _ in range(5):
            err = torch.zeros(1, dtype=torch.int32, device=dev)
            _, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T, err=err)
            torch.cuda.synchronize()
            flagged[0] |= bool(int(err.item()) & _lib.SLP_DEVICE_ERR_TIMEOUT)
            err = torch.zeros(1, dtype=torch.int32, device=dev)
            slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, torch.zeros_like(lse), a.g,
                                    err=err)
            torch.cuda.synchronize()
            flagged[1] |= bool(int(err.item()) & _lib.SLP_DEVICE_ERR_TIMEOUT)
            if all(flagged):
                break
    finally:
        slp.slp_lmhead_set_wait_limit_ns(0)
    assert all(flagged), flagged
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lp, lse = slp.slp_lmhead_forward(a.h, a.W, a.t, a.mask, a.T, err=err)
    dh, dW = slp.slp_lmhead_backward(a.h, a.W, a.t, a.mask, a.T, lse, a.g, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check(a, lp, lse, dh, dW)
    print("one-CTA form OK", flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
