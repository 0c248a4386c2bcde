"""CPU oracle for the Q4_0 x Q8_0 quantized matmul -- TEST INFRASTRUCTURE ONLY.

This package wraps ``q4q_oracle.c`` (plain C99, see its header for the method
and the readings it takes) with ctypes and numpy.  Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import it; the CUDA library
never does, and this package never imports the CUDA library.

Method: "llama.cpp 深度解读" (luoboask.github.io) §2 "量化数据结构 — Q4_0 格式详解"
and §3 "量化矩阵乘法 — 核心算子".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4q_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
# The mutation tests (tests/test_oracle_mutations.py) run the pins against copies
# of q4q_oracle.c with one planted mistake each: Q4Q_ORACLE_SRC names such a copy,
# which is then built into its own library beside it.
if os.environ.get("Q4Q_ORACLE_SRC"):
    _SRC = os.path.abspath(os.environ["Q4Q_ORACLE_SRC"])
    _LIB_PATH = os.path.join(os.path.dirname(_SRC), "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

QK = 32
Q4_0_BYTES = 18
Q8_0_BYTES = 34


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2 -ffp-contract=off -fopenmp)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(os.path.join(_HERE, "q4q_oracle.h")))):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-Wall", "-I" + _HERE, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.orc_fp16_from_f32.restype = ctypes.c_uint16
        lib.orc_fp16_from_f32.argtypes = [ctypes.c_float]
        lib.orc_f32_from_fp16.restype = ctypes.c_float
        lib.orc_f32_from_fp16.argtypes = [ctypes.c_uint16]
        lib.orc_fp16_from_f32_n.argtypes = [P, P, I64]
        lib.orc_f32_from_fp16_n.argtypes = [P, P, I64]
        lib.orc_sizeof_block_q4_0.restype = ctypes.c_size_t
        lib.orc_sizeof_block_q8_0.restype = ctypes.c_size_t
        for name in ("orc_quantize_q4_0", "orc_quantize_q8_0",
                     "orc_dequantize_q4_0", "orc_dequantize_q8_0"):
            getattr(lib, name).argtypes = [P, P, I64, I64]
        lib.orc_vec_dot_q4_0_q8_0.restype = ctypes.c_float
        lib.orc_vec_dot_q4_0_q8_0.argtypes = [I64, P, P]
        lib.orc_block_isums.argtypes = [P, P, I64, I64, I64, P]
        lib.orc_mul_mat.restype = ctypes.c_int
        lib.orc_mul_mat.argtypes = [P, I64, I64, P, I64, I64, P, P, ctypes.c_int]
        lib.orc_mul_mat_q8.restype = ctypes.c_int
        lib.orc_mul_mat_q8.argtypes = [P, I64, I64, P, I64, P, P, ctypes.c_int]
        lib.orc_mul_mat_decoded_f64.argtypes = [P, I64, I64, P, I64, P]
        lib.orc_max_threads.restype = ctypes.c_int
        lib.orc_get_rows_q4_0.restype = ctypes.c_int
        lib.orc_get_rows_q4_0.argtypes = [P, I64, I64, P, I64, P]
        lib.orc_get_rows_q8_0.restype = ctypes.c_int
        lib.orc_get_rows_q8_0.argtypes = [P, I64, I64, P, I64, P]
        lib.orc_silu.restype = ctypes.c_double
        lib.orc_silu.argtypes = [ctypes.c_double]
        lib.orc_gelu.restype = ctypes.c_double
        lib.orc_gelu.argtypes = [ctypes.c_double]
        lib.orc_bias_act.argtypes = [P, P, ctypes.c_int, I64, I64]
        lib.orc_swiglu.argtypes = [P, P, P, I64]
        lib.orc_vec_dot_q8_0_q8_0.restype = ctypes.c_float
        lib.orc_vec_dot_q8_0_q8_0.argtypes = [I64, P, P]
        lib.orc_block_isums_w8.argtypes = [P, P, I64, I64, I64, P]
        lib.orc_mul_mat_w8_q8.restype = ctypes.c_int
        lib.orc_mul_mat_w8_q8.argtypes = [P, I64, I64, P, I64, P, P, ctypes.c_int]
        lib.orc_mul_mat_w8.restype = ctypes.c_int
        lib.orc_mul_mat_w8.argtypes = [P, I64, I64, P, I64, I64, P, P, ctypes.c_int]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


def sizeof_block_q4_0() -> int:
    return int(_load().orc_sizeof_block_q4_0())


def sizeof_block_q8_0() -> int:
    return int(_load().orc_sizeof_block_q8_0())


def max_threads() -> int:
    return int(_load().orc_max_threads())


def fp16_from_f32(x) -> np.ndarray:
    """binary32 -> binary16 bits (uint16), round to nearest even."""
    x = _f32(x)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_fp16_from_f32_n(_ptr(x), _ptr(out), x.size)
    return out


def f32_from_fp16(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().orc_f32_from_fp16_n(_ptr(h), _ptr(out), h.size)
    return out


def quantize_q4_0(src) -> np.ndarray:
    """fp32 [nrows, ncols] -> uint8 [nrows, ncols/32 * 18] (Q4_0 blocks)."""
    src = _f32(src)
    nrows, ncols = src.shape
    assert ncols % QK == 0
    out = np.empty((nrows, ncols // QK * Q4_0_BYTES), dtype=np.uint8)
    _load().orc_quantize_q4_0(_ptr(src), _ptr(out), ncols, nrows)
    return out


def quantize_q8_0(src) -> np.ndarray:
    """fp32 [nrows, ncols] -> uint8 [nrows, ncols/32 * 34] (Q8_0 blocks)."""
    src = _f32(src)
    nrows, ncols = src.shape
    assert ncols % QK == 0
    out = np.empty((nrows, ncols // QK * Q8_0_BYTES), dtype=np.uint8)
    _load().orc_quantize_q8_0(_ptr(src), _ptr(out), ncols, nrows)
    return out


def dequantize_q4_0(blocks, ncols: int) -> np.ndarray:
    blocks = _u8(blocks)
    nrows = blocks.size // (ncols // QK * Q4_0_BYTES)
    out = np.empty((nrows, ncols), dtype=np.float32)
    _load().orc_dequantize_q4_0(_ptr(blocks), _ptr(out), ncols, nrows)
    return out


def dequantize_q8_0(blocks, ncols: int) -> np.ndarray:
    blocks = _u8(blocks)
    nrows = blocks.size // (ncols // QK * Q8_0_BYTES)
    out = np.empty((nrows, ncols), dtype=np.float32)
    _load().orc_dequantize_q8_0(_ptr(blocks), _ptr(out), ncols, nrows)
    return out


def vec_dot_q4_0_q8_0(n: int, x_row, y_row) -> float:
    x_row = _u8(x_row)
    y_row = _u8(y_row)
    return float(_load().orc_vec_dot_q4_0_q8_0(n, _ptr(x_row), _ptr(y_row)))


def block_isums(src0_q4_0, src1_q8_0, ne00: int, ne01: int, ne11: int) -> np.ndarray:
    """int32 [ne11, ne01, ne00/32]: per-block integer dot products."""
    a = _u8(src0_q4_0)
    b = _u8(src1_q8_0)
    out = np.empty((ne11, ne01, ne00 // QK), dtype=np.int32)
    _load().orc_block_isums(_ptr(a), _ptr(b), ne00, ne01, ne11, _ptr(out))
    return out


def mul_mat(src0_q4_0, ne00: int, ne01: int, src1, nthreads: int = 1, with_scale: bool = True):
    """ggml_mul_mat(Q4_0 [ne00, ne01], F32 [ne10, ne11]) -> (dst fp32 [ne11, ne01],
    abs_scale fp64 [ne11, ne01] or None)."""
    a = _u8(src0_q4_0)
    x = _f32(src1)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    ne11, ne10 = x.shape
    dst = np.empty((ne11, ne01), dtype=np.float32)
    scale = np.empty((ne11, ne01), dtype=np.float64) if with_scale else None
    rc = _load().orc_mul_mat(_ptr(a), ne00, ne01, _ptr(x), ne10, ne11, _ptr(dst),
                             _ptr(scale) if with_scale else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle mul_mat: bad shapes")
    return dst, scale


def mul_mat_q8(src0_q4_0, ne00: int, ne01: int, src1_q8_0, ne11: int, nthreads: int = 1):
    a = _u8(src0_q4_0)
    b = _u8(src1_q8_0)
    dst = np.empty((ne11, ne01), dtype=np.float32)
    scale = np.empty((ne11, ne01), dtype=np.float64)
    rc = _load().orc_mul_mat_q8(_ptr(a), ne00, ne01, _ptr(b), ne11, _ptr(dst), _ptr(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle mul_mat_q8: bad shapes")
    return dst, scale


def mul_mat_decoded_f64(src0_q4_0, ne00: int, ne01: int, src1_q8_0, ne11: int) -> np.ndarray:
    a = _u8(src0_q4_0)
    b = _u8(src1_q8_0)
    dst = np.empty((ne11, ne01), dtype=np.float64)
    _load().orc_mul_mat_decoded_f64(_ptr(a), ne00, ne01, _ptr(b), ne11, _ptr(dst))
    return dst


# ------------------------------------------------------------ row gather --

def get_rows(table, ncols: int, ids, kind: str = "q4_0"):
    """ggml_get_rows on a quantized table: fp32 [len(ids), ncols], row i = decode(table row ids[i]).
    Returns (rows, ok): ok is False when some id was out of range (its row is zero)."""
    t = _u8(table)
    idx = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    bpb = Q4_0_BYTES if kind == "q4_0" else Q8_0_BYTES
    nrows = t.size // (ncols // QK * bpb)
    out = np.empty((idx.size, ncols), dtype=np.float32)
    fn = _load().orc_get_rows_q4_0 if kind == "q4_0" else _load().orc_get_rows_q8_0
    rc = fn(_ptr(t), ncols, nrows, _ptr(idx), idx.size, _ptr(out))
    if rc == -1:
        raise ValueError("oracle get_rows: bad shapes")
    return out, rc == 0


# ------------------------------------------------------------- epilogues --

ACT_NONE = 0
ACT_GELU = 1


def silu(x: float) -> float:
    return float(_load().orc_silu(float(x)))


def gelu(x: float) -> float:
    return float(_load().orc_gelu(float(x)))


def bias_act(y, bias=None, act: int = ACT_NONE) -> np.ndarray:
    """fp32 [ne11, ne01]: act(fp32(y + bias)) with bias repeated over the rows of y."""
    out = _f32(y).copy()
    ne11, ne01 = out.shape
    b = _f32(bias) if bias is not None else None
    _load().orc_bias_act(_ptr(out), _ptr(b) if b is not None else None, int(act), ne01, ne11)
    return out


def swiglu(gate, up) -> np.ndarray:
    """fp32(fp32(silu(gate)) * up), elementwise."""
    g = _f32(gate)
    u = _f32(up)
    assert g.shape == u.shape
    out = np.empty(g.shape, dtype=np.float32)
    _load().orc_swiglu(_ptr(g), _ptr(u), _ptr(out), g.size)
    return out


def mul_mat_epilogue(src0_q4_0, ne00: int, ne01: int, src1, bias=None, act: int = ACT_NONE, nthreads: int = 1):
    """act(mul_mat + bias): returns (dst, pre, scale) where pre = fp32(mul_mat + bias)
    (the value the activation sees) and scale the per-element tolerance scale of mul_mat."""
    y, scale = mul_mat(src0_q4_0, ne00, ne01, src1, nthreads=nthreads)
    pre = bias_act(y, bias, ACT_NONE)
    return bias_act(y, bias, act), pre, scale


def mul_mat_swiglu(gate_q4_0, up_q4_0, ne00: int, ne01: int, src1, nthreads: int = 1):
    """silu(gate x) * (up x): returns (dst, g, u, g_scale, u_scale)."""
    g, sg = mul_mat(gate_q4_0, ne00, ne01, src1, nthreads=nthreads)
    u, su = mul_mat(up_q4_0, ne00, ne01, src1, nthreads=nthreads)
    return swiglu(g, u), g, u, sg, su


# ---------------------------------------------------------- Q8_0 weights --

def vec_dot_q8_0_q8_0(n: int, x_row, y_row) -> float:
    x_row = _u8(x_row)
    y_row = _u8(y_row)
    return float(_load().orc_vec_dot_q8_0_q8_0(n, _ptr(x_row), _ptr(y_row)))


def block_isums_w8(src0_q8_0, src1_q8_0, ne00: int, ne01: int, ne11: int) -> np.ndarray:
    """int32 [ne11, ne01, ne00/32]: per-block integer dot products of Q8_0 weights and activations."""
    a = _u8(src0_q8_0)
    b = _u8(src1_q8_0)
    out = np.empty((ne11, ne01, ne00 // QK), dtype=np.int32)
    _load().orc_block_isums_w8(_ptr(a), _ptr(b), ne00, ne01, ne11, _ptr(out))
    return out


def mul_mat_w8(src0_q8_0, ne00: int, ne01: int, src1, nthreads: int = 1):
    """ggml_mul_mat(Q8_0 [ne00, ne01], F32 [ne10, ne11]) -> (dst fp32 [ne11, ne01], scale fp64)."""
    a = _u8(src0_q8_0)
    x = _f32(src1)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    ne11, ne10 = x.shape
    dst = np.empty((ne11, ne01), dtype=np.float32)
    scale = np.empty((ne11, ne01), dtype=np.float64)
    rc = _load().orc_mul_mat_w8(_ptr(a), ne00, ne01, _ptr(x), ne10, ne11, _ptr(dst), _ptr(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle mul_mat_w8: bad shapes")
    return dst, scale


def mul_mat_w8_q8(src0_q8_0, ne00: int, ne01: int, src1_q8_0, ne11: int, nthreads: int = 1):
    a = _u8(src0_q8_0)
    b = _u8(src1_q8_0)
    dst = np.empty((ne11, ne01), dtype=np.float32)
    scale = np.empty((ne11, ne01), dtype=np.float64)
    rc = _load().orc_mul_mat_w8_q8(_ptr(a), ne00, ne01, _ptr(b), ne11, _ptr(dst), _ptr(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle mul_mat_w8_q8: bad shapes")
    return dst, scale
