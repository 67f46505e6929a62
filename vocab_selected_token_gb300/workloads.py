"""Seeded synthetic inputs for the five workloads.

This module only draws random tensors with the shapes and value distributions
of the workloads the source pages discuss (RL micro-batches of a few thousand
to tens of thousands of tokens over 131k-248k-entry vocabularies).  It holds
none of the log-probability arithmetic, so both the CUDA library's tests and
the CPU oracle can be fed from it.

Every tensor comes from one ``torch.Generator`` seeded with the workload's
index (0 tiny, 1 c151k, 2 packed, 3 stability, 4 lmhead), drawn in float32 and
rounded to bfloat16 (round-to-nearest-even) where bfloat16 is asked for.  The
draws are made on the device the caller names; a CUDA generator and a CPU
generator give different (but each reproducible) streams.

Sizes may be overridden (``N=``, ``V=``, ``d=``) to get the same recipe at a
scale the CPU oracle finishes in seconds.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

# name -> (seed, recipe).  The recipe strings are for humans; the generator
# functions below are the definition.
WORKLOADS = {
    "tiny": dict(seed=0, N=256, V=2048, dtype="bf16", T=1.0,
                 recipe="bf16 x~N(0,2^2); t~U[0,V); no mask; g~U(-1,1)"),
    "c151k": dict(seed=1, N=4096, V=151936, dtype="bf16", T=1.0,
                  recipe="bf16 x~N(0,3^2) + 8 at one uniform column per row; "
                         "t = row argmax (p=0.5) else U[0,V); g~U(-1,1)"),
    "packed": dict(seed=2, N=16384, V=248320, dtype="bf16", T=0.7,
                   recipe="bf16 x~N(0,3^2); mask = spans of length U{64..1024}, "
                          "each span on with p=0.3; t~U[0,V); g~U(-1,1)"),
    "stability": dict(seed=3, N=8192, V=131072, dtype="f32", T=1.0,
                      recipe="f32 x~N(0,4^2); each entry +-80 with p=0.01; "
                             "round(0.05N) rows get 1024 distinct -inf columns; "
                             "t~U over finite columns; g~U(-1,1)"),
    "topk": dict(seed=5, N=4096, V=248320, K=128, dtype="bf16", T=1.0, clamp=-10.0,
                 recipe="student bf16 x~N(0,3^2); teacher ids = top-K of x + N(0,1) noise; "
                        "teacher p_k = mass (1-r) r^k / (1-r^K), r=0.95, mass~U(0.85,0.99); "
                        "clamp -10; g~U(-1,1)"),
    "lmhead": dict(seed=4, N=8192, V=151936, d=2560, dtype="bf16", T=1.0,
                   recipe="h bf16~N(0,1) [N,d]; W bf16~N(0,0.02^2) [V,d]; "
                          "t~U[0,V); mask~Bernoulli(0.5); g~U(-1,1)"),
}


@dataclass
class LogitsInputs:
    x: torch.Tensor          # [N, V] bf16 or f32
    t: torch.Tensor          # [N] int32
    mask: torch.Tensor | None  # [N] uint8 or None
    T: float
    g: torch.Tensor          # [N] f32 (upstream gradient of logprob)
    name: str


@dataclass
class TopKInputs:
    x: torch.Tensor          # [N, V] student logits
    ids: torch.Tensor        # [N, K] int32 teacher top-K token ids (distinct per row)
    lt: torch.Tensor         # [N, K] f32 teacher log-probabilities of those ids
    mask: torch.Tensor | None
    T: float
    clamp: float
    g: torch.Tensor          # [N] f32 upstream gradient of the per-token KL
    name: str


@dataclass
class LMHeadInputs:
    h: torch.Tensor          # [N, d] bf16
    W: torch.Tensor          # [V, d] bf16
    t: torch.Tensor          # [N] int32
    mask: torch.Tensor | None
    T: float
    g: torch.Tensor          # [N] f32
    name: str


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def _randn(shape, std, gen, device, row_chunk=1024):
    """float32 N(0, std^2) drawn in row chunks (bounds the float32 temporary)."""
    out = torch.empty(shape, dtype=torch.float32, device=device)
    for r in range(0, shape[0], row_chunk):
        out[r:r + row_chunk].normal_(0.0, std, generator=gen)
    return out


def _to_bf16_chunked(xf: torch.Tensor, row_chunk=1024) -> torch.Tensor:
    out = torch.empty(xf.shape, dtype=torch.bfloat16, device=xf.device)
    for r in range(0, xf.shape[0], row_chunk):
        out[r:r + row_chunk] = xf[r:r + row_chunk].to(torch.bfloat16)
    return out


def _uniform_targets(N, V, gen, device):
    return torch.randint(0, V, (N,), generator=gen, device=device, dtype=torch.int64).to(torch.int32)


def _grad_out(N, gen, device):
    return (torch.rand(N, generator=gen, device=device, dtype=torch.float32) * 2.0 - 1.0)


def span_mask(N: int, p_on: float, lo: int, hi: int, gen, device) -> torch.Tensor:
    """Mask made of consecutive spans with lengths U{lo..hi} (last one cut at N),
    each span switched on with probability p_on: the response spans of packed
    multi-turn sequences."""
    cpu = torch.Generator().manual_seed(int(torch.randint(0, 2**62, (1,), generator=gen, device=device).item()))
    mask = torch.zeros(N, dtype=torch.uint8)
    pos = 0
    while pos < N:
        L = int(torch.randint(lo, hi + 1, (1,), generator=cpu).item())
        on = bool(torch.rand(1, generator=cpu).item() < p_on)
        if on:
            mask[pos:pos + L] = 1
        pos += L
    return mask.to(device)


def make_logits_inputs(name: str, device="cpu", N: int | None = None,
                       V: int | None = None, seed: int | None = None) -> LogitsInputs:
    """Inputs of the logits-input path for workload ``name`` (tiny, c151k,
    packed, stability), optionally at another size with the same recipe."""
    w = WORKLOADS[name]
    N = w["N"] if N is None else int(N)
    V = w["V"] if V is None else int(V)
    gen = _gen(w["seed"] if seed is None else seed, device)
    T = float(w["T"])
    mask = None

    if name == "tiny":
        x = _to_bf16_chunked(_randn((N, V), 2.0, gen, device))
        t = _uniform_targets(N, V, gen, device)
    elif name == "c151k":
        xf = _randn((N, V), 3.0, gen, device)
        spike = torch.randint(0, V, (N,), generator=gen, device=device)
        xf[torch.arange(N, device=device), spike] += 8.0
        x = _to_bf16_chunked(xf)
        del xf
        t_uni = torch.randint(0, V, (N,), generator=gen, device=device)
        use_argmax = torch.rand(N, generator=gen, device=device) < 0.5
        amax = torch.empty(N, dtype=torch.int64, device=device)
        for r in range(0, N, 1024):
            # torch.argmax returns the first (lowest) index among equal maxima
            amax[r:r + 1024] = torch.argmax(x[r:r + 1024], dim=1)
        t = torch.where(use_argmax, amax, t_uni).to(torch.int32)
    elif name == "packed":
        x = _to_bf16_chunked(_randn((N, V), 3.0, gen, device))
        t = _uniform_targets(N, V, gen, device)
        mask = span_mask(N, 0.3, 64, 1024, gen, device)
    elif name == "stability":
        x = _randn((N, V), 4.0, gen, device)
        for r in range(0, N, 1024):
            blk = x[r:r + 1024]
            hit = torch.rand(blk.shape, generator=gen, device=device) < 0.01
            sign = torch.where(torch.rand(blk.shape, generator=gen, device=device) < 0.5, 80.0, -80.0)
            blk[hit] = sign[hit]
        n_inf = int(round(0.05 * N))
        n_cols = min(1024, V - 1)
        rows = torch.randperm(N, generator=gen, device=device)[:n_inf]
        ninf_cols = torch.empty((n_inf, n_cols), dtype=torch.int64, device=device)
        for i in range(n_inf):
            ninf_cols[i] = torch.randperm(V, generator=gen, device=device)[:n_cols]
        if n_inf:
            x[rows.unsqueeze(1).expand(-1, n_cols), ninf_cols] = float("-inf")
        t = _uniform_targets(N, V, gen, device).to(torch.int64)
        # redraw targets that landed on a -inf column until none does
        for _ in range(64):
            bad = torch.isinf(x[torch.arange(N, device=device), t])
            if not bool(bad.any()):
                break
            t = torch.where(bad, torch.randint(0, V, (N,), generator=gen, device=device), t)
        t = t.to(torch.int32)
    else:
        raise ValueError(f"not a logits-input workload: {name}")

    g = _grad_out(N, gen, device)
    return LogitsInputs(x=x, t=t, mask=mask, T=T, g=g, name=name)


def make_lmhead_inputs(name: str = "lmhead", device="cpu", N: int | None = None,
                       V: int | None = None, d: int | None = None,
                       seed: int | None = None, p_mask: float = 0.5) -> LMHeadInputs:
    """Inputs of the fused LM-head path: hidden states, output embedding,
    targets, a Bernoulli(p_mask) loss mask and the upstream gradient."""
    w = WORKLOADS[name]
    N = w["N"] if N is None else int(N)
    V = w["V"] if V is None else int(V)
    d = w["d"] if d is None else int(d)
    gen = _gen(w["seed"] if seed is None else seed, device)
    h = _to_bf16_chunked(_randn((N, d), 1.0, gen, device))
    W = _to_bf16_chunked(_randn((V, d), 0.02, gen, device, row_chunk=8192), row_chunk=8192)
    t = _uniform_targets(N, V, gen, device)
    mask = (torch.rand(N, generator=gen, device=device) < p_mask).to(torch.uint8)
    g = _grad_out(N, gen, device)
    return LMHeadInputs(h=h, W=W, t=t, mask=mask, T=float(w["T"]), g=g, name=name)


def make_topk_inputs(name: str = "topk", device="cpu", N: int | None = None,
                     V: int | None = None, K: int | None = None,
                     seed: int | None = None) -> TopKInputs:
    """Student logits and a synthetic teacher given by its top-K ids and
    log-probabilities (the distillation payload of a top-k forward KL): the
    ids are the top K of the student's logits plus unit Gaussian noise, and the
    probabilities decay geometrically with rank, summing to the teacher's mass
    on its top K."""
    w = WORKLOADS[name]
    N = w["N"] if N is None else int(N)
    V = w["V"] if V is None else int(V)
    K = w["K"] if K is None else int(K)
    gen = _gen(w["seed"] if seed is None else seed, device)
    xf = _randn((N, V), 3.0, gen, device)
    ids = torch.empty((N, K), dtype=torch.int32, device=device)
    for r in range(0, N, 1024):
        blk = xf[r:r + 1024]
        noisy = blk + torch.randn(blk.shape, generator=gen, device=device)
        ids[r:r + 1024] = torch.topk(noisy, K, dim=1).indices.to(torch.int32)
    x = _to_bf16_chunked(xf)
    del xf
    rr = 0.95
    k = torch.arange(K, dtype=torch.float64, device=device)
    shape = (1 - rr) * rr ** k / (1 - rr ** K)
    mass = 0.85 + 0.14 * torch.rand(N, generator=gen, device=device, dtype=torch.float64)
    lt = torch.log(mass[:, None] * shape[None, :]).to(torch.float32)
    g = _grad_out(N, gen, device)
    return TopKInputs(x=x, ids=ids, lt=lt, mask=None, T=float(w["T"]), clamp=float(w["clamp"]),
                      g=g, name=name)
