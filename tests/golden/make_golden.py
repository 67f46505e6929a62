"""Writes tests/golden/oracle_cases.json: small hand-chosen inputs and the CPU
oracle's outputs for them.  Calls only the oracle.  The closed forms that these
cases reduce to are checked in tests/test_golden.py, so the stored values are
pinned to mathematics, not only to the oracle that wrote them.

Run from the repository root:  python -m tests.golden.make_golden
"""

import json
import math
import os

import numpy as np

from oracle import slp_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def f32(a):
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def cases():
    out = []
    # softmax (0.1, 0.2, 0.3, 0.4): logits log(1..4) rounded to float32
    out.append(dict(name="quarters", T=1.0, t=[3, 0],
                    x=f32([[0.0, math.log(2), math.log(3), math.log(4)]] * 2),
                    g=[1.0, -0.5],
                    closed_form_lp=[math.log(0.4), math.log(0.1)], closed_form_tol=2e-7))
    # two classes: log-sigmoid
    out.append(dict(name="two_class", T=0.5, t=[1],
                    x=f32([[1.5, -0.5]]), g=[0.75],
                    closed_form_lp=[-math.log1p(math.exp(4.0))], closed_form_tol=1e-12))
    # one spike of height 8 over zeros, V = 1000, T = 0.8
    V, a, j, T = 1000, 8.0, 123, 0.8
    x = np.zeros((2, V)); x[:, j] = a
    den = math.log(math.exp(a / T) + V - 1)
    out.append(dict(name="spike", T=T, t=[j, 7], x=f32(x), g=[1.0, 1.0],
                    closed_form_lp=[a / T - den, -den], closed_form_tol=1e-12))
    # constant logits: -log V
    out.append(dict(name="uniform", T=0.7, t=[0, 6, 3], x=f32(np.full((3, 7), 2.5)),
                    g=[1.0, -1.0, 0.5],
                    closed_form_lp=[-math.log(7)] * 3, closed_form_tol=1e-13))
    for c in out:
        lp, lse = O.selected_logprob_forward(c["x"], c["t"], None, c["T"])
        gx = O.selected_logprob_backward(c["x"], c["t"], None, c["T"], lse, c["g"])
        c["x"] = c["x"].tolist()
        c["logprob"] = lp.tolist()
        c["lse"] = lse.tolist()
        c["grad_x"] = gx.tolist()
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_cases.json"), "w") as f:
        json.dump({"source": "tests/golden/make_golden.py (CPU oracle only)",
                   "cases": cases()}, f, indent=1)
