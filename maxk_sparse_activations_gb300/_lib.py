"""ctypes loader for librtopk.so (the C ABI declared in include/rtopk.h).

Loading fails loudly: there is no CPU fallback. If the library is missing or
older than its sources it is rebuilt with nvcc first (see build.py).
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

RTOPK_F32 = 0
RTOPK_BF16 = 1

STATUS_NONFINITE = 0x1
STATUS_RANGE = 0x2
STATUS_SAFETY_CAP = 0x4
STATUS_BAD_INDEX = 0x8
STATUS_BAD_EDGE = 0x10

#: every symbol include/rtopk.h declares
EXPORTED = ("rtopk_select", "rtopk_select_stats", "rtopk_select_bucketed", "maxk_forward", "maxk_backward_scatter",
            "maxk_spgemm_forward", "maxk_sspmm_backward", "maxk_sspmm_backward_scatter", "rtopk_status_read",
            "rtopk_strerror", "rtopk_version")


def load(build_if_stale: bool = True) -> ctypes.CDLL:
    """Return the loaded librtopk.so, building it first when stale."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_stale:
            path = _build.build_library()
        else:
            path = _build.LIB
        try:
            lib = ctypes.CDLL(path)
        except OSError as e:
            raise RuntimeError(f"librtopk.so could not be loaded from {path}: {e}. "
                               "Build it with `python -m maxk_sparse_activations_gb300.build`.") from e
        p, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        lib.rtopk_select.argtypes = [p, i64, i32, i32, i32, f32, i32, p, p, p]
        lib.rtopk_select_stats.argtypes = [p, i64, i32, i32, i32, f32, i32, p, p, p, p, p]
        lib.rtopk_select_bucketed.argtypes = [p, i64, i32, i32, i32, i32, f32, i32, p, p, p]
        lib.maxk_forward.argtypes = [p, i64, i32, i32, i32, f32, p, p, p]
        lib.maxk_backward_scatter.argtypes = [p, p, i64, i32, i32, p, p, p]
        lib.maxk_spgemm_forward.argtypes = [p, p, p, i64, i64, p, p, i32, i32, p, p, p]
        lib.maxk_sspmm_backward.argtypes = [p, p, p, i64, i64, p, p, i32, i32, p, p, p]
        lib.maxk_sspmm_backward_scatter.argtypes = [p, p, p, i64, i64, p, p, i32, i32, p, p, p]
        lib.rtopk_status_read.argtypes = [p, p, p]
        lib.rtopk_status_read.restype = ctypes.c_int
        lib.rtopk_strerror.argtypes = [ctypes.c_int]
        lib.rtopk_strerror.restype = ctypes.c_char_p
        lib.rtopk_version.argtypes = []
        for name in ("rtopk_select", "rtopk_select_stats", "rtopk_select_bucketed", "maxk_forward", "maxk_backward_scatter",
                     "maxk_spgemm_forward", "maxk_sspmm_backward", "maxk_sspmm_backward_scatter",
                     "rtopk_version"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def strerror(code: int) -> str:
    return load().rtopk_strerror(int(code)).decode()


def check(code: int, what: str) -> None:
    if code != 0:
        raise RuntimeError(f"{what} failed: {strerror(code)} (code {code})")
