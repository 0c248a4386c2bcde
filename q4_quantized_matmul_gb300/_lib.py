"""ctypes loader for libq4q.so (the CUDA kernels behind the C ABI in include/q4q.h).

There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libq4q.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "q4q.h")

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I64 = ctypes.c_int64
STATUS = ctypes.c_int

_SIGNATURES = {
    "q4q_quantize_q4_0": (STATUS, [P, P, I64, I64, P]),
    "q4q_quantize_q8_0": (STATUS, [P, P, I64, I64, P]),
    "q4q_mul_mat_workspace_size": (STATUS, [I64, I64, I64, ctypes.POINTER(ctypes.c_size_t)]),
    "q4q_mul_mat": (STATUS, [P, I64, I64, P, I64, I64, P, P, ctypes.c_size_t, P]),
    "q4q_mul_mat_ex": (STATUS, [P, I64, I64, P, I64, I64, P, P, ctypes.c_size_t, ctypes.c_uint, P]),
    "q4q_mul_mat_noalloc": (STATUS, [P, I64, I64, P, I64, I64, P, P]),
    "q4q_mul_mat_bias_act": (STATUS, [P, I64, I64, P, I64, I64, P, ctypes.c_int, P, P, ctypes.c_size_t,
                                      ctypes.c_uint, P]),
    "q4q_mul_mat_swiglu_workspace_size": (STATUS, [I64, I64, I64, ctypes.POINTER(ctypes.c_size_t)]),
    "q4q_mul_mat_swiglu": (STATUS, [P, P, I64, I64, P, I64, I64, P, P, ctypes.c_size_t, ctypes.c_uint, P]),
    "q4q_get_rows_q4_0": (STATUS, [P, I64, I64, P, I64, P, P]),
    "q4q_get_rows_q8_0": (STATUS, [P, I64, I64, P, I64, P, P]),
    "q4q_mul_mat_q8_0_workspace_size": (STATUS, [I64, I64, I64, ctypes.POINTER(ctypes.c_size_t)]),
    "q4q_mul_mat_q8_0": (STATUS, [P, I64, I64, P, I64, I64, P, P, ctypes.c_size_t, ctypes.c_uint, P]),
    "q4q_debug_block_isums_q8_0": (STATUS, [P, P, I64, I64, I64, ctypes.c_int, P, P, ctypes.c_size_t, P]),
    "q4q_mul_mat_group_workspace_size": (STATUS, [ctypes.c_int, ctypes.POINTER(I64), I64, I64,
                                                  ctypes.POINTER(ctypes.c_size_t)]),
    "q4q_mul_mat_group": (STATUS, [ctypes.c_int, ctypes.POINTER(P), ctypes.POINTER(I64), I64, P, I64, I64,
                                   ctypes.POINTER(P), P, ctypes.c_size_t, ctypes.c_uint, P]),
    "q4q_debug_workspace_size": (STATUS, [I64, I64, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "q4q_debug_block_isums": (STATUS, [P, P, I64, I64, I64, ctypes.c_int, P, P, ctypes.c_size_t, P]),
    "q4q_device_status": (STATUS, [ctypes.POINTER(ctypes.c_int)]),
    "q4q_debug_wait_timeout": (STATUS, [ctypes.c_uint64, P]),
    "q4q_debug_mul_mat_timeout": (STATUS, [P, I64, I64, P, I64, P, P, ctypes.c_size_t, ctypes.c_int,
                                           ctypes.c_uint64, P]),
    "q4q_debug_mul_mat_path": (STATUS, [P, I64, I64, P, I64, P, P, ctypes.c_size_t, ctypes.c_int, P]),
    "q4q_debug_mul_mat_path_workspace_size": (STATUS, [I64, I64, I64, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "q4q_debug_gemv_plan": (STATUS, [I64, I64, I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.POINTER(I64)]),
    "q4q_debug_mma_splits": (STATUS, [I64, I64, I64, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]),
    "q4q_mul_mat_chain_workspace_size": (STATUS, [ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "q4q_mul_mat_chain": (STATUS, [P, ctypes.c_int, I64, P, ctypes.c_size_t, ctypes.c_uint, P]),
    "q4q_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "q4q_version": (ctypes.c_int, []),
}


def declared_entry_points(header: str = HEADER):
    """Names of the functions include/q4q.h declares with Q4Q_API."""
    with open(header, encoding="utf-8") as f:
        text = f.read()
    return re.findall(r"^Q4Q_API\s+[^(;]*?\b(q4q_\w+)\s*\(", text, flags=re.M)


def load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libq4q.so is not built (%s); run __graft_entry__.build() first" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib
