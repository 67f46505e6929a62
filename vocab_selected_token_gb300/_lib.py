"""ctypes loader for the in-tree libslp.so.  There is no fallback: if the
library has not been built, every call raises."""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libslp.so")

SLP_BF16 = 0
SLP_F32 = 1
SLP_OK = 0
SLP_ERR_INVALID_ARG = 1
SLP_ERR_UNSUPPORTED = 2
SLP_ERR_MISALIGNED = 3
SLP_ERR_WORKSPACE = 4
SLP_ERR_CUDA = 5
SLP_DATA_ERR_TARGET = 1
SLP_DEVICE_ERR_TIMEOUT = 2
SLP_DEVICE_ERR_BOUNDS = 4

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_int = ctypes.c_int
_sz = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/slp.h
SIGNATURES = {
    "slp_forward": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp, _vp, _vp]),
    "slp_backward": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp, _vp, _i64,
                            _vp, _vp]),
    "slp_forward_entropy": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp, _vp,
                                   _vp, _vp]),
    "slp_backward_entropy": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp, _vp,
                                    _vp, _vp, _i64, _vp, _vp]),
    "slp_topk_kl_forward": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _i64, _vp, _f32, _f32,
                                   _vp, _vp, _vp, _vp, _vp, _vp]),
    "slp_topk_kl_backward": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _i64, _vp, _f32, _f32,
                                    _vp, _vp, _vp, _i64, _vp, _vp]),
    "slp_forward_backward": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp, _vp,
                                    _vp, _i64, _vp, _vp]),
    "slp_forward_backward_entropy": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _f32, _vp,
                                            _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp]),
    "slp_forward_backward_host_workspace_size": (_sz, [_i64, _i64, _int, _i64]),
    "slp_forward_backward_host": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp,
                                         _vp, _vp, _i64, _i64, _vp, _sz, _vp, _vp]),
    "slp_lmhead_workspace_size": (_sz, [_i64, _i64, _i64]),
    "slp_lmhead_forward_workspace_size": (_sz, [_i64, _i64, _i64]),
    "slp_lmhead_workspace_size_max": (_sz, [_i64, _i64, _i64]),
    "slp_lmhead_workspace_size_min": (_sz, [_i64, _i64, _i64]),
    "slp_lmhead_forward": (_int, [_vp, _vp, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp, _vp,
                                  _sz, _vp, _vp]),
    "slp_lmhead_backward": (_int, [_vp, _vp, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp, _vp,
                                   _vp, _vp, _sz, _vp, _vp]),
    "slp_lmhead_forward_noalloc": (_int, [_vp, _vp, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp,
                                          _vp, _vp]),
    "slp_lmhead_backward_accumulate": (_int, [_vp, _vp, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp,
                                              _vp, _vp, _vp, _sz, _vp, _vp]),
    "slp_lmhead_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "slp_bounds_check_selftest": (_int, [_vp, _vp, _vp]),
    "slp_status_string": (ctypes.c_char_p, [_int]),
}

_lib = None


class SlpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} (status {status})")


def load() -> ctypes.CDLL:
    """Load libslp.so once.  Raises if it is missing: build it with
    ``python -m vocab_selected_token_gb300.build``."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libslp.so is not built ({LIB_PATH}); run "
                               "`python -m vocab_selected_token_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().slp_status_string(int(status)).decode()


def call(name: str, *args) -> None:
    st = getattr(load(), name)(*args)
    if st != SLP_OK:
        raise SlpError(name, st)
