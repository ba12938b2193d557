"""ctypes loader of libqmla.so (the in-tree C-ABI library).

There is no fallback: if the library is missing or fails to load, importing
the binding raises, so nothing can silently run another implementation."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmla.so")

_lib = None

# exported symbols, as declared in include/qmla.h
SYMBOLS = ("qmla_block_bytes", "qmla_append", "qmla_append_advance",
           "qmla_decode_workspace_bytes", "qmla_decode", "qmla_decode_multi",
           "qmla_decode_noalloc", "qmla_decode_timeout_test", "qmla_decode_step_layout",
           "qmla_decode_step_workspace_bytes", "qmla_decode_step", "qmla_read_status",
           "qmla_error_string")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"libqmla.so not found at {path}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    L.qmla_block_bytes.argtypes = [ctypes.c_int]
    L.qmla_block_bytes.restype = sz
    L.qmla_append.argtypes = [ctypes.c_int, P, i64, P, i32, P, i32, i32, P, P, P, P]
    L.qmla_append.restype = ctypes.c_int
    L.qmla_append_advance.argtypes = [ctypes.c_int, P, i64, P, i32, P, i32, i32, P, P, P, P]
    L.qmla_append_advance.restype = ctypes.c_int
    L.qmla_decode_workspace_bytes.argtypes = [ctypes.c_int, i32, i32, i32]
    L.qmla_decode_workspace_bytes.restype = sz
    L.qmla_decode.argtypes = [ctypes.c_int, P, i64, P, i32, P, i32, i32, i32, P, P, f32, P, P, P,
                              sz, P, P]
    L.qmla_decode.restype = ctypes.c_int
    L.qmla_decode_multi.argtypes = [ctypes.c_int, P, i64, P, i32, P, i32, i32, i32, i32, P, P,
                                    f32, P, P, P, sz, P, P]
    L.qmla_decode_multi.restype = ctypes.c_int
    L.qmla_decode_noalloc.argtypes = [ctypes.c_int, P, i64, P, i32, P, i32, i32, i32, P, P, f32,
                                      P, P, P, P]
    L.qmla_decode_noalloc.restype = ctypes.c_int
    L.qmla_decode_timeout_test.argtypes = L.qmla_decode.argtypes
    L.qmla_decode_timeout_test.restype = ctypes.c_int
    L.qmla_decode_step_layout.argtypes = [i32, i32, i32, ctypes.POINTER(sz)]
    L.qmla_decode_step_layout.restype = ctypes.c_int
    L.qmla_decode_step_workspace_bytes.argtypes = [ctypes.c_int, i32, i32, i32, i32]
    L.qmla_decode_step_workspace_bytes.restype = sz
    L.qmla_decode_step.argtypes = [ctypes.c_int, P, i64, P, i32, P, i32, i32, i32, i32, P, f32, P,
                                   P, sz, P, P]
    L.qmla_decode_step.restype = ctypes.c_int
    L.qmla_read_status.argtypes = [P, P]
    L.qmla_read_status.restype = ctypes.c_int
    L.qmla_error_string.argtypes = [ctypes.c_int]
    L.qmla_error_string.restype = ctypes.c_char_p
    _lib = L
    return L
