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
    # the backward needs the larger workspace
    assert b(FAKE, FAKE, N, V, d, FAKE, None, 1.0, FAKE, FAKE, FAKE, FAKE, FAKE, need_b - 1,
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


def test_fused_entropy_binding_checks_before_the_library():
    """slp_forward_backward_entropy's binding rejects bad outputs (overlap
    with x, wrong shape or dtype) and bad vectors before any library call."""
    import torch

    import vocab_selected_token_gb300 as slp
    x = torch.zeros(4, 8, dtype=torch.bfloat16)
    t = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError):
        slp.slp_forward_backward_entropy(x, t, None, 1.0, grad_x=x)
    with pytest.raises(ValueError):
        slp.slp_forward_backward_entropy(x, t, None, 1.0, grad_x=torch.zeros(4, 8))
    with pytest.raises(ValueError):
        slp.slp_forward_backward_entropy(x, t, None, 1.0, grad_out=torch.zeros(3))
    with pytest.raises(ValueError):
        slp.slp_forward_backward_entropy(x, t.long(), None, 1.0)


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
