"""CPU-only: the C-ABI library loads, exports every function include/slp.h
declares, and rejects bad arguments before touching the device."""

import ctypes
import os
import re

import pytest

from vocab_selected_token_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**\s*(slp_\w+)\s*\(",
                             src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from vocab_selected_token_gb300 import build
    build.build()
    return _lib.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("slp_forward", "slp_backward", "slp_lmhead_workspace_size",
              "slp_lmhead_forward", "slp_lmhead_backward", "slp_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature"


def test_status_strings(lib):
    assert _lib.status_string(0) == "ok"
    assert "invalid" in _lib.status_string(1)
    assert _lib.status_string(99) == "unknown status"


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first


@pytest.mark.parametrize("args,expect", [
    # (x, dtype, N, V, ld, t, mask, T, lp, lse, err, stream)
    ((FAKE, 0, -1, 10, 10, FAKE, None, 1.0, FAKE, FAKE, None, None), _lib.SLP_ERR_INVALID_ARG),
    ((FAKE, 0, 4, 0, 10, FAKE, None, 1.0, FAKE, FAKE, None, None), _lib.SLP_ERR_INVALID_ARG),
    ((FAKE, 0, 4, 10, 9, FAKE, None, 1.0, FAKE, FAKE, None, None), _lib.SLP_ERR_INVALID_ARG),
    ((FAKE, 7, 4, 10, 10, FAKE, None, 1.0, FAKE, FAKE, None, None), _lib.SLP_ERR_INVALID_ARG),
    ((FAKE, 0, 4, 10, 10, FAKE, None, 0.0, FAKE, FAKE, None, None), _lib.SLP_ERR_INVALID_ARG),
    ((FAKE, 0, 4, 10, 10, FAKE, None, float("nan"), FAKE, FAKE, None, None), _lib.SLP_ERR_INVALID_ARG),
    ((FAKE, 0, 4, 10, 10, FAKE, None, float("inf"), FAKE, FAKE, None, None), _lib.SLP_ERR_INVALID_ARG),
    ((None, 0, 4, 10, 10, FAKE, None, 1.0, FAKE, FAKE, None, None), _lib.SLP_ERR_INVALID_ARG),
    ((FAKE, 0, 4, 10, 10, None, None, 1.0, FAKE, FAKE, None, None), _lib.SLP_ERR_INVALID_ARG),
    ((FAKE, 0, 4, 10, 10, FAKE, None, 1.0, None, FAKE, None, None), _lib.SLP_ERR_INVALID_ARG),
    ((None, 0, 0, 10, 10, None, None, 1.0, None, None, None, None), _lib.SLP_OK),  # N = 0: no-op
])
def test_forward_argument_errors(lib, args, expect):
    assert lib.slp_forward(*args) == expect


def test_backward_argument_errors(lib):
    # ld_grad < V
    assert lib.slp_backward(FAKE, 0, 4, 10, 10, FAKE, None, 1.0, FAKE, FAKE, FAKE, 9, None,
                            None) == _lib.SLP_ERR_INVALID_ARG
    # missing lse
    assert lib.slp_backward(FAKE, 0, 4, 10, 10, FAKE, None, 1.0, None, FAKE, FAKE, 10, None,
                            None) == _lib.SLP_ERR_INVALID_ARG
    assert lib.slp_backward(None, 1, 0, 10, 10, None, None, 1.0, None, None, None, 10, None,
                            None) == _lib.SLP_OK


def test_forward_backward_entropy_argument_errors(lib):
    f = lib.slp_forward_backward_entropy
    # (x, dtype, N, V, ld, t, mask, T, g, gH, lp, lse, H, gx, ld_grad, err, stream)
    assert f(FAKE, 0, 4, 10, 10, FAKE, None, 1.0, None, None, FAKE, FAKE, FAKE, FAKE, 9, None,
             None) == _lib.SLP_ERR_INVALID_ARG                                  # ld_grad < V
    assert f(FAKE, 0, 4, 10, 10, FAKE, None, 1.0, None, None, FAKE, FAKE, None, FAKE, 10, None,
             None) == _lib.SLP_ERR_INVALID_ARG                                  # no entropy out
    assert f(FAKE, 0, 4, 10, 10, FAKE, None, -1.0, None, None, FAKE, FAKE, FAKE, FAKE, 10, None,
             None) == _lib.SLP_ERR_INVALID_ARG                                  # T <= 0
    assert f(None, 1, 0, 10, 10, None, None, 1.0, None, None, None, None, None, None, 10, None,
             None) == _lib.SLP_OK                                               # N = 0: no-op


def test_lmhead_argument_errors(lib):
    N, V, d = 64, 1000, 128
    need_b = lib.slp_lmhead_workspace_size(N, V, d)
    need = lib.slp_lmhead_forward_workspace_size(N, V, d)
    assert 0 < need <= need_b
    assert lib.slp_lmhead_workspace_size(-1, V, d) == 0
    assert lib.slp_lmhead_forward_workspace_size(N, 0, d) == 0
    f = lib.slp_lmhead_forward
    # d not a multiple of 64
    assert f(FAKE, FAKE, N, V, 100, FAKE, None, 1.0, FAKE, FAKE, FAKE, 1 << 40, None,
             None) == _lib.SLP_ERR_UNSUPPORTED
    # misaligned h
    assert f(ctypes.c_void_p(0x1008), FAKE, N, V, d, FAKE, None, 1.0, FAKE, FAKE, FAKE, need,
             None, None) == _lib.SLP_ERR_MISALIGNED
    # workspace too small / missing
    assert f(FAKE, FAKE, N, V, d, FAKE, None, 1.0, FAKE, FAKE, FAKE, need - 1, None,
             None) == _lib.SLP_ERR_WORKSPACE
    assert f(FAKE, FAKE, N, V, d, FAKE, None, 1.0, FAKE, FAKE, None, need, None,
             None) == _lib.SLP_ERR_WORKSPACE
    # bad temperature
    assert f(FAKE, FAKE, N, V, d, FAKE, None, -1.0, FAKE, FAKE, FAKE, need, None,
             None) == _lib.SLP_ERR_INVALID_ARG
    b = lib.slp_lmhead_backward
    assert b(FAKE, FAKE, N, V, d, FAKE, None, 1.0, FAKE, FAKE, None, FAKE, FAKE, need_b, None,
             None) == _lib.SLP_ERR_INVALID_ARG
    assert b(FAKE, FAKE, N, V, d, FAKE, None, 1.0, FAKE, FAKE, ctypes.c_void_p(0x1002), FAKE,
             FAKE, need_b, None, None) == _lib.SLP_ERR_MISALIGNED
    # the backward needs at least its minimum workspace (16384-column chunks)
    need_min = lib.slp_lmhead_workspace_size_min(N, V, d)
    assert need <= need_min <= need_b
    assert b(FAKE, FAKE, N, V, d, FAKE, None, 1.0, FAKE, FAKE, FAKE, FAKE, FAKE, need_min - 1,
             None, None) == _lib.SLP_ERR_WORKSPACE


def test_product_path_has_no_oracle_import():
    pkg = os.path.join(ROOT, "vocab_selected_token_gb300")
    pat = re.compile(r"^\s*(from|import)\s+(\.\.)?oracle\b|slp_oracle", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                assert not pat.search(open(os.path.join(dirpath, f)).read()), f


def test_host_streaming_argument_errors(lib):
    """slp_forward_backward_host rejects bad arguments before any CUDA call."""
    f = lib.slp_forward_backward_host
    # (x, dtype, N, V, ld, t, mask, T, g, lp, lse, gx, ld_grad, rows_per_chunk, ws, ws_bytes, err, stream)
    good = [FAKE, 0, 4, 16, 16, FAKE, None, 1.0, FAKE, FAKE, FAKE, FAKE, 16, 0, FAKE, 1 << 20,
            None, None]
    for i, bad in ((2, -1), (4, 8), (7, 0.0), (8, None), (12, 8), (1, 7), (3, 0)):
        a = list(good)
        a[i] = bad
        assert f(*a) == _lib.SLP_ERR_INVALID_ARG, (i, bad)
    a = list(good)
    a[2] = 0
    assert f(*a) == _lib.SLP_OK  # N = 0: nothing to do


def test_host_streaming_workspace_size(lib):
    ws = lib.slp_forward_backward_host_workspace_size
    assert ws(-1, 10, 0, 0) == 0 and ws(10, 0, 0, 0) == 0 and ws(10, 10, 5, 0) == 0
    V = 151936
    row = V * 2

    def slot(r, esize=2):  # one chunk of logits and one of gradient
        return 2 * ((r * V * esize + 255) // 256 * 256)

    def vectors(n):  # t, g, mask, logprob, lse of every row
        return sum((n * b + 255) // 256 * 256 for b in (4, 4, 1, 4, 4))

    R = (64 << 20) // row  # default plan: equal chunks of about 64 MB of logits
    assert ws(R, V, 0, 0) == vectors(R) + slot(R)                 # one chunk: one slot
    assert ws(2 * R, V, 0, 0) == vectors(2 * R) + 2 * slot(R)
    assert ws(4096, V, 0, 0) == vectors(4096) + 3 * slot(R)       # three slots in the ring
    assert ws(100, V, 0, 0) == vectors(100) + slot(100)           # fewer rows than a chunk
    assert ws(100, V, 1, 25) == vectors(100) + 3 * slot(25, 4)   # equal chunks of 25 rows


def test_binding_refuses_overlapping_outputs():
    """The binding rejects an output that shares memory with an input before
    anything reaches the library (slp.h: outputs must not overlap inputs)."""
    import torch

    import vocab_selected_token_gb300 as slp
    x = torch.zeros(4, 8)
    with pytest.raises(ValueError):
        slp._check_disjoint("grad_x", x, x)
    with pytest.raises(ValueError):
        slp._check_disjoint("grad_x", x[1:], x)
    slp._check_disjoint("grad_x", torch.zeros(4, 8), x)
    slp._check_disjoint("dW", torch.zeros(3, 2), None, torch.zeros(5))


@pytest.fixture
def no_library_call(monkeypatch):
    """Makes any call into libslp fail the test: the binding's checks must
    refuse bad tensors before the library sees a pointer."""
    from vocab_selected_token_gb300 import _lib

    def refuse(name, *args):
        raise AssertionError(f"{name} reached the library")

    monkeypatch.setattr(_lib, "call", refuse)


CUDA_ONLY = "must be CUDA tensors"  # the last check: well-formed CPU tensors end there


def test_fused_entropy_binding_checks_before_the_library(no_library_call):
    """slp_forward_backward_entropy's binding rejects bad outputs (overlap
    with x, wrong shape or dtype) and bad vectors before any library call."""
    import torch

    import vocab_selected_token_gb300 as slp
    x = torch.zeros(4, 8, dtype=torch.bfloat16)
    t = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="overlap"):
        slp.slp_forward_backward_entropy(x, t, None, 1.0, grad_x=x)
    with pytest.raises(ValueError, match="grad_x must be"):
        slp.slp_forward_backward_entropy(x, t, None, 1.0, grad_x=torch.zeros(4, 8))
    with pytest.raises(ValueError, match="grad_out"):
        slp.slp_forward_backward_entropy(x, t, None, 1.0, grad_out=torch.zeros(3))
    with pytest.raises(ValueError, match="t must be"):
        slp.slp_forward_backward_entropy(x, t.long(), None, 1.0)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        slp.slp_forward_backward_entropy(x, t, None, 1.0)


def _bad_grad_x(x):
    """grad_x tensors the library must never be handed for logits x [N, V]."""
    import torch
    N, V = x.shape
    wide = torch.zeros(N, 2 * V, dtype=x.dtype)
    return [
        ("grad_x must be", torch.zeros(N, V + 1, dtype=x.dtype)),       # too many columns
        ("grad_x must be", torch.zeros(N - 1, V, dtype=x.dtype)),       # too few rows
        ("grad_x must be", torch.zeros(N, V, dtype=torch.float64)),     # wrong dtype
        ("grad_x must be", torch.zeros(N * V, dtype=x.dtype)),          # wrong rank
        ("unit column stride", wide[:, ::2]),                           # strided columns
        ("must not overlap", torch.zeros(V, dtype=x.dtype).expand(N, V)),  # rows alias
        ("overlap", x),                                                 # in place of x
    ]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_logits_backward_bindings_check_grad_x_before_the_library(no_library_call, dtype):
    """Every logits-path binding that takes a caller's grad_x checks its shape,
    dtype, column stride, row stride and overlap with x before the call
    (slp_backward, slp_backward_entropy, slp_topk_kl_backward,
    slp_forward_backward, slp_forward_backward_entropy); a well-formed CPU
    grad_x gets as far as the device check."""
    import torch

    import vocab_selected_token_gb300 as slp
    N, V, K = 4, 8, 3
    x = torch.zeros(N, V, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32)
    t = torch.zeros(N, dtype=torch.int32)
    v = torch.zeros(N)
    ids = torch.zeros(N, K, dtype=torch.int32)
    lt = torch.zeros(N, K)
    calls = {
        "slp_backward": lambda gx: slp.slp_backward(x, t, None, 1.0, v, v, grad_x=gx),
        "slp_backward_entropy": lambda gx: slp.slp_backward_entropy(x, t, None, 1.0, v, v, v, v,
                                                                    grad_x=gx),
        "slp_topk_kl_backward": lambda gx: slp.slp_topk_kl_backward(x, ids, lt, None, 1.0, -10.0,
                                                                    v, v, grad_x=gx),
        "slp_forward_backward": lambda gx: slp.slp_forward_backward(x, t, None, 1.0, v,
                                                                    grad_x=gx),
        "slp_forward_backward_entropy": lambda gx: slp.slp_forward_backward_entropy(
            x, t, None, 1.0, v, v, grad_x=gx),
    }
    for name, call in calls.items():
        for why, gx in _bad_grad_x(x):
            with pytest.raises(ValueError, match=why):
                call(gx)
        with pytest.raises(ValueError, match=CUDA_ONLY):
            call(torch.zeros(N, V, dtype=x.dtype))
        with pytest.raises(ValueError, match=CUDA_ONLY):
            call(torch.zeros(N, V + 5, dtype=x.dtype)[:, :V])  # padded rows are fine


def test_lmhead_backward_bindings_check_outputs_before_the_library(no_library_call):
    """slp_lmhead_backward checks dh [N, d] and dW [V, d] (bf16, contiguous,
    disjoint from h, W and each other), slp_lmhead_backward_accumulate checks
    dh and its float32 dW accumulator, and both check the workspace, before
    the library is called."""
    import torch

    import vocab_selected_token_gb300 as slp
    N, V, d = 4, 16, 64
    h = torch.zeros(N, d, dtype=torch.bfloat16)
    W = torch.zeros(V, d, dtype=torch.bfloat16)
    t = torch.zeros(N, dtype=torch.int32)
    v = torch.zeros(N)
    dh_ok = torch.zeros(N, d, dtype=torch.bfloat16)
    dW_ok = torch.zeros(V, d, dtype=torch.bfloat16)
    ws = torch.zeros(slp.slp_lmhead_workspace_size(N, V, d), dtype=torch.uint8)

    def bwd(dh=dh_ok, dW=dW_ok, ws=ws):
        return slp.slp_lmhead_backward(h, W, t, None, 1.0, v, v, dh=dh, dW=dW, ws=ws)

    bad_dh = [torch.zeros(N, d + 64, dtype=torch.bfloat16), torch.zeros(N + 1, d, dtype=torch.bfloat16),
              torch.zeros(N, d), torch.zeros(N, 2 * d, dtype=torch.bfloat16)[:, ::2]]
    bad_dW = [torch.zeros(V - 1, d, dtype=torch.bfloat16), torch.zeros(V, d),
              torch.zeros(d, V, dtype=torch.bfloat16).t()]
    for dh in bad_dh:
        with pytest.raises(ValueError, match="dh must be"):
            bwd(dh=dh)
    for dW in bad_dW:
        with pytest.raises(ValueError, match="dW must be"):
            bwd(dW=dW)
    with pytest.raises(ValueError, match="overlap"):
        bwd(dW=W)
    with pytest.raises(ValueError, match="overlap"):
        bwd(dh=h)
    with pytest.raises(ValueError, match="ws must be"):
        bwd(ws=torch.zeros(2 * ws.numel(), dtype=torch.uint8)[::2])
    with pytest.raises(ValueError, match=CUDA_ONLY):
        bwd()

    acc_ok = torch.zeros(V, d)

    def acc(dW_accum=acc_ok, dh=dh_ok):
        return slp.slp_lmhead_backward_accumulate(h, W, t, None, 1.0, v, v, dW_accum, dh=dh,
                                                  ws=ws)

    for bad in (torch.zeros(V, d, dtype=torch.bfloat16), torch.zeros(V + 1, d),
                torch.zeros(d, V).t()):
        with pytest.raises(ValueError, match="dW_accum must be"):
            acc(dW_accum=bad)
    for dh in bad_dh:
        with pytest.raises(ValueError, match="dh must be"):
            acc(dh=dh)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        acc()


def test_lmhead_workspace_bytes_count_the_element_size(monkeypatch):
    """A caller's workspace is passed with its size in bytes, whatever its
    dtype, and a non-contiguous one is refused (its numel would overstate the
    memory the library may write)."""
    import torch

    import vocab_selected_token_gb300 as slp
    monkeypatch.setattr(slp, "slp_lmhead_workspace_size", lambda N, V, d: 1)
    ws, nbytes = slp._workspace(1, 1, 64, torch.zeros(100, dtype=torch.float32), None)
    assert nbytes == 400
    ws, nbytes = slp._workspace(1, 1, 64, torch.zeros(100, dtype=torch.uint8), None)
    assert nbytes == 100
    with pytest.raises(ValueError, match="ws must be"):
        slp._workspace(1, 1, 64, torch.zeros(10, 10, dtype=torch.uint8)[:, :5], None)


def test_error_word_and_device_checks(no_library_call):
    """The error word must be an int32 tensor; CPU tensors never reach the
    library (the no-allocation forward included)."""
    import torch

    import vocab_selected_token_gb300 as slp
    N, V, d = 4, 16, 64
    x = torch.zeros(N, V)
    t = torch.zeros(N, dtype=torch.int32)
    with pytest.raises(ValueError, match="err must be"):
        slp.slp_forward(x, t, err=torch.zeros(1, dtype=torch.int64))
    with pytest.raises(ValueError, match=CUDA_ONLY):
        slp.slp_forward(x, t, err=torch.zeros(1, dtype=torch.int32))
    h = torch.zeros(N, d, dtype=torch.bfloat16)
    W = torch.zeros(V, d, dtype=torch.bfloat16)
    lp = torch.zeros(N)
    with pytest.raises(ValueError, match="lse must be"):
        slp.slp_lmhead_forward_noalloc(h, W, t, None, 1.0, lp, torch.zeros(N + 1))
    with pytest.raises(ValueError, match=CUDA_ONLY):
        slp.slp_lmhead_forward_noalloc(h, W, t, None, 1.0, lp, torch.zeros(N))


def test_lmhead_workspace_size_max(lib):
    """The whole-vocabulary workspace is at least the default one, equal to it
    when the vocabulary fits one default chunk, and 0 for invalid sizes."""
    big = lib.slp_lmhead_workspace_size_max(8192, 151936, 2560)
    dflt = lib.slp_lmhead_workspace_size(8192, 151936, 2560)
    assert big > dflt > lib.slp_lmhead_forward_workspace_size(8192, 151936, 2560)
    assert lib.slp_lmhead_workspace_size_max(300, 60000, 256) == \
        lib.slp_lmhead_workspace_size(300, 60000, 256)
    assert lib.slp_lmhead_workspace_size_max(-1, 100, 64) == 0
    assert lib.slp_lmhead_workspace_size_max(10, 100, 0) == 0


def test_lmhead_workspace_size_min(lib):
    """The 16384-column workspace is well below the default one, never above
    it (for a vocabulary within one minimum chunk only its split-K partials
    are smaller), still holds the forward's workspace, and is 0 for invalid
    sizes."""
    small = lib.slp_lmhead_workspace_size_min(8192, 151936, 2560)
    dflt = lib.slp_lmhead_workspace_size(8192, 151936, 2560)
    assert lib.slp_lmhead_forward_workspace_size(8192, 151936, 2560) <= small < dflt
    assert small < 0.4 * dflt  # a quarter of the dz buffer, fewer split-K partials
    assert lib.slp_lmhead_forward_workspace_size(300, 16000, 256) <= \
        lib.slp_lmhead_workspace_size_min(300, 16000, 256) <= \
        lib.slp_lmhead_workspace_size(300, 16000, 256)
    assert lib.slp_lmhead_workspace_size_min(-1, 100, 64) == 0
