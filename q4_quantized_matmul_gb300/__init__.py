"""Q4_0 x Q8_0 quantized matmul for GB300 (sm_103a).

A thin binding over the C ABI of libq4q.so (include/q4q.h).  Each function has
the name of the C entry point it calls and only marshals arguments: torch CUDA
tensors in, pointers and sizes out, the current torch CUDA stream as the
stream.  Every step of the computation runs in the library's CUDA kernels.

The operation is ggml_mul_mat(Q4_0 weights, F32 activations) as described in
"llama.cpp 深度解读" (luoboask.github.io) §2 and §3.
"""
from __future__ import annotations

import ctypes
import functools
from typing import Optional

import torch

from . import _lib

__all__ = [
    "Q4QError", "q4q_quantize_q4_0", "q4q_quantize_q8_0", "q4q_mul_mat_workspace_size",
    "q4q_mul_mat", "q4q_debug_block_isums", "q4q_debug_workspace_size", "Q4Q_MUL_MAT_PDL",
    "q4q_mul_mat_noalloc", "Q4Q_NOALLOC_SCRATCH_BYTES", "q4q_device_status", "q4q_status_string",
    "q4q_version", "q4_0_row_bytes", "q8_0_row_bytes", "mul_mat_host",
    "Q4Q_ACT_NONE", "Q4Q_ACT_GELU", "q4q_mul_mat_bias_act", "q4q_mul_mat_swiglu_workspace_size",
    "q4q_mul_mat_swiglu", "q4q_get_rows_q4_0", "q4q_get_rows_q8_0", "q4q_mul_mat_q8_0_workspace_size",
    "q4q_mul_mat_q8_0", "q4q_debug_block_isums_q8_0", "Q4Q_GROUP_MAX", "q4q_mul_mat_group_workspace_size",
    "q4q_mul_mat_group", "q4q_debug_wait_timeout",
]

QK = 32
Q4_0_BYTES = 18
Q8_0_BYTES = 34

STATUS_NAMES = {0: "Q4Q_OK", 1: "Q4Q_ERR_NULL", 2: "Q4Q_ERR_SHAPE", 3: "Q4Q_ERR_ALIGN",
                4: "Q4Q_ERR_WORKSPACE", 5: "Q4Q_ERR_CUDA", 6: "Q4Q_ERR_TIMEOUT", 7: "Q4Q_ERR_ARG"}


class Q4QError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (fn, STATUS_NAMES.get(status, status), q4q_status_string(status)))


def _check(fn: str, status: int):
    if status != 0:
        raise Q4QError(fn, status)


def _first_cuda_device(values):
    for v in values:
        if isinstance(v, torch.Tensor) and v.is_cuda:
            return v.device
        if isinstance(v, (list, tuple)):
            d = _first_cuda_device(v)
            if d is not None:
                return d
    return None


def _on_tensor_device(fn):
    """Run a wrapper with the device of its first CUDA tensor argument current: the
    library plans for, allocates on and launches on the current device (and the
    default stream is that device's current stream)."""
    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        dev = _first_cuda_device(list(args) + list(kwargs.values()))
        if dev is None:
            return fn(*args, **kwargs)
        with torch.cuda.device(dev):
            return fn(*args, **kwargs)
    return wrapper


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return stream


def _dev(t: torch.Tensor, name: str, min_bytes: int = 0):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if t.numel() * t.element_size() < min_bytes:
        raise ValueError("%s holds %d bytes, the call reads or writes %d" % (
            name, t.numel() * t.element_size(), min_bytes))
    return ctypes.c_void_p(t.data_ptr())


def q4_0_row_bytes(ne00: int) -> int:
    return ne00 // QK * Q4_0_BYTES


def q8_0_row_bytes(ne00: int) -> int:
    return ne00 // QK * Q8_0_BYTES


def q4q_version() -> int:
    return int(_lib.load().q4q_version())


def q4q_status_string(status: int) -> str:
    return _lib.load().q4q_status_string(int(status)).decode()


@_on_tensor_device
def _quantize(fn: str, src: torch.Tensor, dst: Optional[torch.Tensor], row_bytes, stream):
    if src.dtype != torch.float32 or src.dim() != 2:
        raise TypeError("src must be a 2-D float32 tensor")
    nrows, ncols = src.shape
    if dst is None:
        dst = torch.empty((nrows, row_bytes(ncols)), dtype=torch.uint8, device=src.device)
    _check(fn, getattr(_lib.load(), fn)(_dev(src, "src"), _dev(dst, "dst", nrows * row_bytes(ncols)), ncols, nrows,
                                         _stream(stream)))
    return dst


def q4q_quantize_q4_0(src: torch.Tensor, dst: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """fp32 [nrows, ncols] -> uint8 [nrows, ncols/32*18] Q4_0 blocks."""
    return _quantize("q4q_quantize_q4_0", src, dst, q4_0_row_bytes, stream)


def q4q_quantize_q8_0(src: torch.Tensor, dst: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """fp32 [nrows, ncols] -> uint8 [nrows, ncols/32*34] Q8_0 blocks."""
    return _quantize("q4q_quantize_q8_0", src, dst, q8_0_row_bytes, stream)


def q4q_mul_mat_workspace_size(ne00: int, ne01: int, ne11: int) -> int:
    n = ctypes.c_size_t(0)
    _check("q4q_mul_mat_workspace_size", _lib.load().q4q_mul_mat_workspace_size(ne00, ne01, ne11, ctypes.byref(n)))
    return int(n.value)


@_on_tensor_device
def q4q_mul_mat(src0: torch.Tensor, ne00: int, ne01: int, src1: torch.Tensor,
                dst: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                stream=None, flags: int = 0) -> torch.Tensor:
    """ggml_mul_mat(Q4_0 src0 [ne00, ne01], F32 src1 [ne00, ne11]) -> F32 [ne11, ne01].

    src0: uint8 CUDA tensor holding ne01 * ne00/32 Q4_0 blocks; src1: float32
    [ne11, ne00]; dst (optional): float32 [ne11, ne01]; workspace (optional):
    uint8 tensor of at least q4q_mul_mat_workspace_size(ne00, ne01, ne11) bytes.
    flags != 0 calls q4q_mul_mat_ex (Q4Q_MUL_MAT_PDL = 1).
    """
    if src1.dtype != torch.float32:
        raise TypeError("src1 must be float32")
    x = src1.reshape(-1, src1.shape[-1]) if src1.dim() != 2 else src1
    ne11, ne10 = x.shape
    if dst is None:
        dst = torch.empty((ne11, ne01), dtype=torch.float32, device=x.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is None:
        need = q4q_mul_mat_workspace_size(ne00, ne01, ne11) if ne01 * ne11 > 0 else 0
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    if workspace is not None and workspace.numel() > 0:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    if ne01 * ne11 == 0:
        return dst
    lib = _lib.load()
    w_ptr = _dev(src0, "src0", ne01 * q4_0_row_bytes(ne00))
    d_ptr = _dev(dst, "dst", 4 * ne01 * ne11)
    if flags:
        _check("q4q_mul_mat_ex", lib.q4q_mul_mat_ex(w_ptr, ne00, ne01, _dev(x, "src1"), ne10, ne11,
                                                   d_ptr, ws_ptr, ws_bytes, int(flags), _stream(stream)))
    else:
        _check("q4q_mul_mat", lib.q4q_mul_mat(w_ptr, ne00, ne01, _dev(x, "src1"), ne10, ne11,
                                             d_ptr, ws_ptr, ws_bytes, _stream(stream)))
    return dst


Q4Q_MUL_MAT_PDL = 1
Q4Q_NOALLOC_SCRATCH_BYTES = 8 << 20


@_on_tensor_device
def q4q_mul_mat_noalloc(src0: torch.Tensor, ne00: int, ne01: int, src1: torch.Tensor,
                        dst: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q4q_mul_mat without a workspace, for callers that cannot allocate device
    memory: the library's own static scratch array (Q4Q_NOALLOC_SCRATCH_BYTES per
    GPU) stands in for it.  Calls that overlap on the GPU share that array and
    race; larger problems raise Q4QError (Q4Q_ERR_WORKSPACE)."""
    if src1.dtype != torch.float32:
        raise TypeError("src1 must be float32")
    x = src1.reshape(-1, src1.shape[-1]) if src1.dim() != 2 else src1
    ne11, ne10 = x.shape
    if dst is None:
        dst = torch.empty((ne11, ne01), dtype=torch.float32, device=x.device)
    if ne01 * ne11 == 0:
        return dst
    _check("q4q_mul_mat_noalloc", _lib.load().q4q_mul_mat_noalloc(_dev(src0, "src0", ne01 * q4_0_row_bytes(ne00)),
                                                                 ne00, ne01, _dev(x, "src1"), ne10, ne11,
                                                                 _dev(dst, "dst", 4 * ne01 * ne11), _stream(stream)))
    return dst


def q4q_debug_workspace_size(ne00: int, ne11: int, path: int) -> int:
    n = ctypes.c_size_t(0)
    _check("q4q_debug_workspace_size", _lib.load().q4q_debug_workspace_size(ne00, ne11, int(path), ctypes.byref(n)))
    return int(n.value)


@_on_tensor_device
def q4q_debug_block_isums(src0: torch.Tensor, src1_q8_0: torch.Tensor, ne00: int, ne01: int, ne11: int,
                          path: int = 0, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """int32 [ne11, ne01, ne00/32] per-block integer sums from the device routine of `path`."""
    if out is None:
        out = torch.empty((ne11, ne01, ne00 // QK), dtype=torch.int32, device=src0.device)
    need = q4q_debug_workspace_size(ne00, ne11, path)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=src0.device)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check("q4q_debug_block_isums",
           _lib.load().q4q_debug_block_isums(_dev(src0, "src0", ne01 * q4_0_row_bytes(ne00)),
                                             _dev(src1_q8_0, "src1_q8_0", ne11 * q8_0_row_bytes(ne00)), ne00, ne01,
                                             ne11, int(path), _dev(out, "out", 4 * ne11 * ne01 * (ne00 // QK)),
                                             ws_ptr, ws_bytes, _stream(stream)))
    return out


def q4q_device_status() -> int:
    """Synchronize the device and return (and clear) the device-side status word."""
    st = ctypes.c_int(0)
    _check("q4q_device_status", _lib.load().q4q_device_status(ctypes.byref(st)))
    return int(st.value)


def mul_mat_host(src0: torch.Tensor, ne00: int, ne01: int, src1_host: torch.Tensor, dst_host: torch.Tensor,
                 src1_dev: torch.Tensor, dst_dev: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """q4q_mul_mat with host activations and a host result: pinned host -> device
    copy of src1, the C-ABI call, device -> pinned host copy of dst, all on one stream."""
    src1_dev.copy_(src1_host, non_blocking=True)
    q4q_mul_mat(src0, ne00, ne01, src1_dev, dst=dst_dev, workspace=workspace, stream=stream)
    dst_host.copy_(dst_dev, non_blocking=True)
    return dst_host


# ------------------------------------------------------ next to the matmul --

Q4Q_ACT_NONE = 0
Q4Q_ACT_GELU = 1


def _acts_2d(src1: torch.Tensor) -> torch.Tensor:
    if src1.dtype != torch.float32:
        raise TypeError("src1 must be float32")
    return src1.reshape(-1, src1.shape[-1]) if src1.dim() != 2 else src1


def _workspace(need: int, workspace: Optional[torch.Tensor], device):
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if workspace is not None and workspace.numel() > 0:
        return _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    return None, 0


@_on_tensor_device
def q4q_mul_mat_bias_act(src0: torch.Tensor, ne00: int, ne01: int, src1: torch.Tensor,
                         bias: Optional[torch.Tensor] = None, act: int = Q4Q_ACT_NONE,
                         dst: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                         stream=None, flags: int = 0) -> torch.Tensor:
    """act(ggml_mul_mat(Q4_0 src0, F32 src1) + bias) -> F32 [ne11, ne01]; bias fp32 [ne01] or None."""
    x = _acts_2d(src1)
    ne11, ne10 = x.shape
    if dst is None:
        dst = torch.empty((ne11, ne01), dtype=torch.float32, device=x.device)
    if ne01 * ne11 == 0:
        return dst
    if bias is not None and (bias.dtype != torch.float32 or bias.numel() != ne01):
        raise ValueError("bias must be float32 with ne01 elements")
    ws_ptr, ws_bytes = _workspace(q4q_mul_mat_workspace_size(ne00, ne01, ne11), workspace, x.device)
    _check("q4q_mul_mat_bias_act", _lib.load().q4q_mul_mat_bias_act(
        _dev(src0, "src0", ne01 * q4_0_row_bytes(ne00)), ne00, ne01, _dev(x, "src1"), ne10, ne11,
        _dev(bias, "bias", 4 * ne01) if bias is not None else None, int(act), _dev(dst, "dst", 4 * ne01 * ne11),
        ws_ptr, ws_bytes, int(flags), _stream(stream)))
    return dst


def q4q_mul_mat_swiglu_workspace_size(ne00: int, ne01: int, ne11: int) -> int:
    n = ctypes.c_size_t(0)
    _check("q4q_mul_mat_swiglu_workspace_size",
           _lib.load().q4q_mul_mat_swiglu_workspace_size(ne00, ne01, ne11, ctypes.byref(n)))
    return int(n.value)


@_on_tensor_device
def q4q_mul_mat_swiglu(gate: torch.Tensor, up: torch.Tensor, ne00: int, ne01: int, src1: torch.Tensor,
                       dst: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                       stream=None, flags: int = 0) -> torch.Tensor:
    """silu(ggml_mul_mat(gate, src1)) * ggml_mul_mat(up, src1) -> F32 [ne11, ne01] (Q4_0 gate and up)."""
    x = _acts_2d(src1)
    ne11, ne10 = x.shape
    if dst is None:
        dst = torch.empty((ne11, ne01), dtype=torch.float32, device=x.device)
    if ne01 * ne11 == 0:
        return dst
    ws_ptr, ws_bytes = _workspace(q4q_mul_mat_swiglu_workspace_size(ne00, ne01, ne11), workspace, x.device)
    nbytes = ne01 * q4_0_row_bytes(ne00)
    _check("q4q_mul_mat_swiglu", _lib.load().q4q_mul_mat_swiglu(
        _dev(gate, "gate", nbytes), _dev(up, "up", nbytes), ne00, ne01, _dev(x, "src1"), ne10, ne11,
        _dev(dst, "dst", 4 * ne01 * ne11), ws_ptr, ws_bytes, int(flags), _stream(stream)))
    return dst


@_on_tensor_device
def _get_rows(fn: str, row_bytes, src0: torch.Tensor, ne00: int, ne01: int, ids: Optional[torch.Tensor],
              n_ids: Optional[int], dst: Optional[torch.Tensor], stream) -> torch.Tensor:
    if ids is not None:
        if ids.dtype != torch.int32:
            raise TypeError("ids must be int32")
        n_ids = ids.numel()
    elif n_ids is None:
        n_ids = ne01
    if dst is None:
        dst = torch.empty((n_ids, ne00), dtype=torch.float32, device=src0.device)
    if n_ids == 0:
        return dst
    _check(fn, getattr(_lib.load(), fn)(_dev(src0, "src0", ne01 * row_bytes(ne00)), ne00, ne01,
                                         _dev(ids, "ids", 4 * n_ids) if ids is not None else None, n_ids,
                                         _dev(dst, "dst", 4 * n_ids * ne00), _stream(stream)))
    return dst


def q4q_get_rows_q4_0(src0: torch.Tensor, ne00: int, ne01: int, ids: Optional[torch.Tensor] = None,
                      n_ids: Optional[int] = None, dst: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """ggml_get_rows on a Q4_0 table [ne01 rows of ne00]: fp32 [n_ids, ne00]; ids None = rows 0..n_ids-1."""
    return _get_rows("q4q_get_rows_q4_0", q4_0_row_bytes, src0, ne00, ne01, ids, n_ids, dst, stream)


def q4q_get_rows_q8_0(src0: torch.Tensor, ne00: int, ne01: int, ids: Optional[torch.Tensor] = None,
                      n_ids: Optional[int] = None, dst: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """ggml_get_rows on a Q8_0 table [ne01 rows of ne00]: fp32 [n_ids, ne00]; ids None = rows 0..n_ids-1."""
    return _get_rows("q4q_get_rows_q8_0", q8_0_row_bytes, src0, ne00, ne01, ids, n_ids, dst, stream)


def q4q_mul_mat_q8_0_workspace_size(ne00: int, ne01: int, ne11: int) -> int:
    n = ctypes.c_size_t(0)
    _check("q4q_mul_mat_q8_0_workspace_size",
           _lib.load().q4q_mul_mat_q8_0_workspace_size(ne00, ne01, ne11, ctypes.byref(n)))
    return int(n.value)


@_on_tensor_device
def q4q_mul_mat_q8_0(src0: torch.Tensor, ne00: int, ne01: int, src1: torch.Tensor,
                     dst: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                     stream=None, flags: int = 0) -> torch.Tensor:
    """ggml_mul_mat(Q8_0 src0 [ne00, ne01], F32 src1 [ne00, ne11]) -> F32 [ne11, ne01]."""
    x = _acts_2d(src1)
    ne11, ne10 = x.shape
    if dst is None:
        dst = torch.empty((ne11, ne01), dtype=torch.float32, device=x.device)
    if ne01 * ne11 == 0:
        return dst
    ws_ptr, ws_bytes = _workspace(q4q_mul_mat_q8_0_workspace_size(ne00, ne01, ne11), workspace, x.device)
    _check("q4q_mul_mat_q8_0", _lib.load().q4q_mul_mat_q8_0(
        _dev(src0, "src0", ne01 * q8_0_row_bytes(ne00)), ne00, ne01, _dev(x, "src1"), ne10, ne11,
        _dev(dst, "dst", 4 * ne01 * ne11), ws_ptr, ws_bytes, int(flags), _stream(stream)))
    return dst


@_on_tensor_device
def q4q_debug_block_isums_q8_0(src0_q8_0: torch.Tensor, src1_q8_0: torch.Tensor, ne00: int, ne01: int, ne11: int,
                               path: int = 0, out: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """int32 [ne11, ne01, ne00/32] block sums of Q8_0 weights x Q8_0 activations from the device
    routine of `path` (0 = GEMV, 1 = tensor-core GEMM)."""
    if out is None:
        out = torch.empty((ne11, ne01, ne00 // QK), dtype=torch.int32, device=src0_q8_0.device)
    need = q4q_debug_workspace_size(ne00, ne11, path)
    ws_ptr, ws_bytes = _workspace(need, workspace, src0_q8_0.device)
    _check("q4q_debug_block_isums_q8_0", _lib.load().q4q_debug_block_isums_q8_0(
        _dev(src0_q8_0, "src0_q8_0", ne01 * q8_0_row_bytes(ne00)),
        _dev(src1_q8_0, "src1_q8_0", ne11 * q8_0_row_bytes(ne00)), ne00, ne01, ne11, int(path),
        _dev(out, "out", 4 * ne11 * ne01 * (ne00 // QK)), ws_ptr, ws_bytes, _stream(stream)))
    return out


Q4Q_GROUP_MAX = 4


def q4q_mul_mat_group_workspace_size(ne01s, ne00: int, ne11: int) -> int:
    n = len(ne01s)
    arr = (ctypes.c_int64 * max(n, 1))(*ne01s)
    out = ctypes.c_size_t(0)
    _check("q4q_mul_mat_group_workspace_size",
           _lib.load().q4q_mul_mat_group_workspace_size(n, arr, ne00, ne11, ctypes.byref(out)))
    return int(out.value)


@_on_tensor_device
def q4q_mul_mat_group(src0s, ne01s, ne00: int, src1: torch.Tensor, dsts=None,
                      workspace: Optional[torch.Tensor] = None, stream=None, flags: int = 0):
    """[ggml_mul_mat(src0s[m] (Q4_0 [ne00, ne01s[m]]), src1) for m] in one call: F32 [ne11, ne01s[m]] each."""
    x = _acts_2d(src1)
    ne11, ne10 = x.shape
    n = len(src0s)
    if n != len(ne01s):
        raise ValueError("one row count per matrix")
    if dsts is None:
        dsts = [torch.empty((ne11, r), dtype=torch.float32, device=x.device) for r in ne01s]
    if ne11 == 0 or n == 0:
        return dsts
    ws_ptr, ws_bytes = _workspace(q4q_mul_mat_group_workspace_size(ne01s, ne00, ne11), workspace, x.device)
    ptrs = (ctypes.c_void_p * n)(*[_dev(w, "src0", r * q4_0_row_bytes(ne00)).value for w, r in zip(src0s, ne01s)])
    outs = (ctypes.c_void_p * n)(*[_dev(d, "dst", 4 * r * ne11).value for d, r in zip(dsts, ne01s)])
    rows = (ctypes.c_int64 * n)(*ne01s)
    _check("q4q_mul_mat_group", _lib.load().q4q_mul_mat_group(n, ptrs, rows, ne00, _dev(x, "src1"), ne10, ne11, outs,
                                                             ws_ptr, ws_bytes, int(flags), _stream(stream)))
    return dsts


def q4q_debug_wait_timeout(limit_ns: int, stream=None) -> None:
    """Run the library's bounded-wait failure path on its own: one wait that nothing
    completes, given up after limit_ns; q4q_device_status() then reports Q4Q_ERR_TIMEOUT (6)."""
    _check("q4q_debug_wait_timeout", _lib.load().q4q_debug_wait_timeout(int(limit_ns), _stream(stream)))


def q4q_debug_mul_mat_path_workspace_size(ne00: int, ne01: int, ne11: int, path: int) -> int:
    n = ctypes.c_size_t(0)
    _check("q4q_debug_mul_mat_path_workspace_size",
           _lib.load().q4q_debug_mul_mat_path_workspace_size(ne00, ne01, ne11, int(path), ctypes.byref(n)))
    return n.value


@_on_tensor_device
def q4q_debug_mul_mat_path(src0: torch.Tensor, ne00: int, ne01: int, src1: torch.Tensor, path: int,
                           dst: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    """q4q_mul_mat on one named path (0 = GEMV, 1 = tensor-core GEMM, 3 = warp-MMA
    kernel), whatever q4q_mul_mat would pick for the shape; workspace defaults to what
    the path plans its split-K for."""
    x = _acts_2d(src1)
    ne11, ne10 = x.shape
    if dst is None:
        dst = torch.empty((ne11, ne01), dtype=torch.float32, device=x.device)
    need = q4q_debug_mul_mat_path_workspace_size(ne00, ne01, ne11, path) if workspace is None else 0
    ws_ptr, ws_bytes = _workspace(need, workspace, x.device)
    _check("q4q_debug_mul_mat_path", _lib.load().q4q_debug_mul_mat_path(
        _dev(src0, "src0", ne01 * q4_0_row_bytes(ne00)), ne00, ne01, _dev(x, "src1"), ne11,
        _dev(dst, "dst", 4 * ne01 * ne11), ws_ptr, ws_bytes, int(path), _stream(stream)))
    return dst


@_on_tensor_device
def q4q_debug_mul_mat_timeout(src0: torch.Tensor, ne00: int, ne01: int, src1: torch.Tensor, path: int,
                              limit_ns: int, dst: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Run the matmul kernel of `path` (0 = GEMV, 1 = tensor-core GEMM, 2 = two-link chain,
    3 = warp-MMA kernel) with one hand-off left out in its first CTA and every wait
    bounded by limit_ns: the waits run out, q4q_device_status() then reports
    Q4Q_ERR_TIMEOUT (6), and dst is incomplete."""
    x = _acts_2d(src1)
    ne11, ne10 = x.shape
    if dst is None:
        dst = torch.empty((ne11, ne01), dtype=torch.float32, device=x.device)
    need = {1: q4q_mul_mat_workspace_size(ne00, ne01, ne11) if path == 1 else 0,
            2: q4q_mul_mat_chain_workspace_size(2) if path == 2 else 0,
            3: q4q_mul_mat_workspace_size(ne00, ne01, ne11) if path == 3 else 0}.get(path, 0)
    ws_ptr, ws_bytes = _workspace(need, workspace, x.device)
    _check("q4q_debug_mul_mat_timeout", _lib.load().q4q_debug_mul_mat_timeout(
        _dev(src0, "src0", ne01 * q4_0_row_bytes(ne00)), ne00, ne01, _dev(x, "src1"), ne11,
        _dev(dst, "dst", 4 * ne01 * ne11), ws_ptr, ws_bytes, int(path), int(limit_ns), _stream(stream)))
    return dst


# --------------------------------------------------- chains of projections --

Q4Q_CHAIN_MAX = 64


class ChainLink(ctypes.Structure):
    """q4q_chain_link of include/q4q.h."""
    _fields_ = [("src0", ctypes.c_void_p), ("ne00", ctypes.c_int64), ("ne01", ctypes.c_int64),
                ("src1", ctypes.c_void_p), ("dst", ctypes.c_void_p)]


def q4q_mul_mat_chain_workspace_size(n: int) -> int:
    out = ctypes.c_size_t(0)
    _check("q4q_mul_mat_chain_workspace_size", _lib.load().q4q_mul_mat_chain_workspace_size(int(n), ctypes.byref(out)))
    return int(out.value)


def chain_links(links):
    """ctypes array of q4q_chain_link from (src0, ne00, ne01, src1, dst) tuples of CUDA tensors."""
    arr = (ChainLink * len(links))()
    for i, (w, ne00, ne01, x, y) in enumerate(links):
        arr[i] = ChainLink(_dev(w, "src0", ne01 * q4_0_row_bytes(ne00)).value, ne00, ne01,
                           _dev(x, "src1", 4 * ne00).value, _dev(y, "dst", 4 * ne01).value)
    return arr


@_on_tensor_device
def q4q_mul_mat_chain(links, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Run a chain of one-token projections in one launch: for each (src0, ne00, ne01,
    src1, dst) in order, dst = ggml_mul_mat(src0, src1); a link's src1 may be an
    earlier link's dst.  src0: uint8 Q4_0 blocks, src1: float32 [ne00], dst: float32 [ne01]."""
    n = len(links)
    arr = chain_links(links)
    if workspace is None:
        workspace = torch.empty(q4q_mul_mat_chain_workspace_size(n), dtype=torch.uint8, device=links[0][0].device)
    _check("q4q_mul_mat_chain", _lib.load().q4q_mul_mat_chain(arr, n, 1, _dev(workspace, "workspace"),
                                                             workspace.numel(), 0, _stream(stream)))
