"""CPU-only: the seeded generators produce the stated shapes, dtypes and
structure, reproducibly."""

import numpy as np
import torch

from vocab_selected_token_gb300 import workloads as W


def test_tiny_shapes_and_reproducible():
    a = W.make_logits_inputs("tiny")
    b = W.make_logits_inputs("tiny")
    assert a.x.shape == (256, 2048) and a.x.dtype == torch.bfloat16
    assert a.t.dtype == torch.int32 and a.mask is None
    assert torch.equal(a.x, b.x) and torch.equal(a.t, b.t) and torch.equal(a.g, b.g)
    assert float(a.x.float().std()) > 1.8 and float(a.x.float().std()) < 2.2
    assert int(a.t.min()) >= 0 and int(a.t.max()) < 2048
    assert float(a.g.abs().max()) <= 1.0


def test_c151k_recipe_small():
    a = W.make_logits_inputs("c151k", N=64, V=4096)
    am = torch.argmax(a.x, dim=1).to(torch.int32)
    frac = float((a.t == am).float().mean())
    assert 0.3 < frac < 0.7           # about half the targets are the row argmax


def test_packed_mask_spans():
    a = W.make_logits_inputs("packed", N=8192, V=64)
    m = a.mask.numpy().astype(np.int8)
    edges = np.flatnonzero(np.diff(np.concatenate([[0], m, [0]])))
    runs = edges[1::2] - edges[::2]
    assert m.mean() > 0.1 and m.mean() < 0.5
    assert runs.min() >= 64 or edges[0] == 0 or edges[-1] == 8192
    assert a.T == 0.7


def test_stability_recipe_small():
    a = W.make_logits_inputs("stability", N=200, V=2048)
    x = a.x
    assert x.dtype == torch.float32
    ninf_rows = torch.isinf(x).any(dim=1) & (x == float("-inf")).any(dim=1)
    assert int(ninf_rows.sum()) == 10
    assert int((x == float("-inf")).sum(dim=1).max()) == 1024
    xt = x[torch.arange(200), a.t.long()]
    assert torch.isfinite(xt).all()
    assert float((x.abs() == 80).float().mean()) > 0.005


def test_lmhead_small():
    a = W.make_lmhead_inputs(N=64, V=300, d=128)
    assert a.h.shape == (64, 128) and a.W.shape == (300, 128)
    assert a.h.dtype == torch.bfloat16 and a.W.dtype == torch.bfloat16
    assert a.mask.dtype == torch.uint8

