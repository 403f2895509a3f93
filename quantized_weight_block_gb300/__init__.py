"""Python binding of the GB300 packed quantized-weight decoder (``libndq.so``).

Argument marshalling only: every decode step runs in the library's CUDA
kernels.  The ``ndq_*`` functions mirror the C ABI in ``include/ndq.h`` one
to one (plain integers and pointers); ``dequantize_packed`` and
``dequantize_packed_batched`` are conveniences that take torch CUDA tensors
and the current torch stream.  There is no CPU fallback: importing this
module fails if the library has not been built
(``python -m quantized_weight_block_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

LIB_PATH = _build.LIB

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m quantized_weight_block_gb300.build` "
                      "(there is no CPU fallback)")

_lib = ctypes.CDLL(LIB_PATH)

# ---- constants mirrored from include/ndq.h --------------------------------
NDQ_OK = 0
STATUS = {
    0: "NDQ_OK", 1: "NDQ_ERR_NULL", 2: "NDQ_ERR_UNKNOWN_FORMAT", 3: "NDQ_ERR_UNSUPPORTED_FORMAT",
    4: "NDQ_ERR_BAD_RANK", 5: "NDQ_ERR_NEGATIVE_DIM", 6: "NDQ_ERR_NOT_BLOCK_ALIGNED",
    7: "NDQ_ERR_LENGTH_MISMATCH", 8: "NDQ_ERR_OVERFLOW", 9: "NDQ_ERR_BAD_DTYPE", 10: "NDQ_ERR_WORKSPACE",
    11: "NDQ_ERR_CUDA", 12: "NDQ_ERR_DEVICE_FAULT", 13: "NDQ_ERR_BAD_COUNT", 14: "NDQ_ERR_TOO_MANY_TENSORS",
}
NDQ_FLOAT, NDQ_FLOAT16, NDQ_DOUBLE, NDQ_BFLOAT16 = 1, 10, 11, 16
NDQ_MAX_RANK = 8
NDQ_NUM_FORMATS = 36
NDQ_NOALLOC_MAX_TENSORS = 1024


class NdqError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        self.name = STATUS.get(status, str(status))
        msg = _lib.ndq_status_string(status).decode()
        super().__init__(f"{self.name}: {msg}" + (f" ({what})" if what else ""))


class ndq_tensor_desc(ctypes.Structure):
    _fields_ = [
        ("format_id", ctypes.c_int32), ("ndim", ctypes.c_int32), ("shape", ctypes.c_int64 * NDQ_MAX_RANK),
        ("out_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32), ("x", ctypes.c_void_p),
        ("x_len", ctypes.c_uint64), ("y", ctypes.c_void_p),
    ]


class ndq_matmul_desc(ctypes.Structure):
    _fields_ = [
        ("format_id", ctypes.c_int32), ("reserved", ctypes.c_int32), ("n", ctypes.c_int64), ("w", ctypes.c_void_p),
        ("w_len", ctypes.c_uint64), ("y", ctypes.c_void_p),
    ]


_c = ctypes
_lib.ndq_format_from_name.argtypes = [_c.c_char_p]
_lib.ndq_format_from_name.restype = _c.c_int
_lib.ndq_format_name.argtypes = [_c.c_int]
_lib.ndq_format_name.restype = _c.c_char_p
_lib.ndq_format_geometry.argtypes = [_c.c_int, _c.POINTER(_c.c_int), _c.POINTER(_c.c_int)]
_lib.ndq_format_supported.argtypes = [_c.c_int]
_lib.ndq_status_string.argtypes = [_c.c_int]
_lib.ndq_status_string.restype = _c.c_char_p
_lib.ndq_payload_geometry.argtypes = [_c.c_int, _c.POINTER(_c.c_int64), _c.c_int, _c.c_uint64,
                                      _c.POINTER(_c.c_uint64), _c.POINTER(_c.c_uint64), _c.POINTER(_c.c_uint64)]
_lib.ndq_dequantize_packed.argtypes = [_c.c_int, _c.POINTER(_c.c_int64), _c.c_int, _c.c_int, _c.c_void_p,
                                       _c.c_size_t, _c.c_void_p, _c.c_void_p]
_lib.ndq_batched_workspace_bytes.argtypes = [_c.c_int]
_lib.ndq_batched_workspace_bytes.restype = _c.c_size_t
_lib.ndq_dequantize_packed_batched.argtypes = [_c.POINTER(ndq_tensor_desc), _c.c_int, _c.c_void_p, _c.c_size_t,
                                               _c.c_void_p]
_lib.ndq_get_device_fault.argtypes = [_c.POINTER(_c.c_uint32)]
_lib.ndq_test_withhold_copy.argtypes = [_c.c_int64, _c.c_uint32]
_lib.ndq_dequantize_packed_batched_noalloc.argtypes = [_c.POINTER(ndq_tensor_desc), _c.c_int, _c.c_void_p]
_lib.ndq_matmul_packed.argtypes = [_c.c_int, _c.c_int64, _c.c_int64, _c.c_void_p, _c.c_size_t, _c.c_void_p,
                                   _c.c_int64, _c.c_int, _c.c_int, _c.c_void_p, _c.c_void_p]
_lib.ndq_matmul_packed_batched.argtypes = [_c.POINTER(ndq_matmul_desc), _c.c_int, _c.c_int64, _c.c_void_p,
                                           _c.c_int64, _c.c_int, _c.c_int, _c.c_void_p]

# Every symbol the header declares (checked by the CPU tests).
EXPORTS = (
    "ndq_format_from_name", "ndq_format_name", "ndq_format_geometry", "ndq_format_supported",
    "ndq_status_string", "ndq_payload_geometry", "ndq_dequantize_packed", "ndq_batched_workspace_bytes",
    "ndq_dequantize_packed_batched", "ndq_get_device_fault", "ndq_dequantize_packed_batched_noalloc",
    "ndq_matmul_packed", "ndq_test_withhold_copy", "ndq_matmul_packed_batched",
)


# ---- raw C ABI (same names, plain integers / pointers) --------------------
def ndq_format_from_name(name: str) -> int:
    return _lib.ndq_format_from_name(name.encode() if name is not None else None)


def ndq_format_name(format_id: int) -> str | None:
    r = _lib.ndq_format_name(format_id)
    return r.decode() if r is not None else None


def ndq_format_geometry(format_id: int) -> tuple[int, int]:
    B, S = _c.c_int(), _c.c_int()
    rc = _lib.ndq_format_geometry(format_id, _c.byref(B), _c.byref(S))
    if rc:
        raise NdqError(rc)
    return B.value, S.value


def ndq_format_supported(format_id: int) -> int:
    return _lib.ndq_format_supported(format_id)


def ndq_status_string(status: int) -> str:
    return _lib.ndq_status_string(status).decode()


def _shape(shape):
    s = [int(d) for d in shape]
    return (_c.c_int64 * max(1, len(s)))(*s), len(s)


def ndq_payload_geometry(format_id: int, shape, x_len: int) -> tuple[int, int, int]:
    sa, nd = _shape(shape)
    nb, ne, ndv = _c.c_uint64(), _c.c_uint64(), _c.c_uint64()
    rc = _lib.ndq_payload_geometry(format_id, sa, nd, x_len, _c.byref(nb), _c.byref(ne), _c.byref(ndv))
    if rc:
        raise NdqError(rc)
    return nb.value, ne.value, ndv.value


def ndq_dequantize_packed(format_id: int, shape, out_dtype: int, x_ptr: int, x_len: int, y_ptr: int,
                          stream: int = 0) -> int:
    """Raw call; returns the status code (0 on success)."""
    sa, nd = _shape(shape)
    return _lib.ndq_dequantize_packed(format_id, sa, nd, out_dtype, x_ptr, x_len, y_ptr, stream)


def ndq_batched_workspace_bytes(n: int) -> int:
    return _lib.ndq_batched_workspace_bytes(n)


def ndq_dequantize_packed_batched(descs, workspace_ptr: int, ws_bytes: int, stream: int = 0) -> int:
    """Raw call over a sequence of ndq_tensor_desc; returns the status code."""
    arr = (ndq_tensor_desc * max(1, len(descs)))(*descs)
    return _lib.ndq_dequantize_packed_batched(arr, len(descs), workspace_ptr, ws_bytes, stream)


def ndq_dequantize_packed_batched_noalloc(descs, stream: int = 0) -> int:
    """Raw call of the no-allocation batched decode (launch table held in the
    library's own device array); returns the status code."""
    arr = (ndq_tensor_desc * max(1, len(descs)))(*descs)
    return _lib.ndq_dequantize_packed_batched_noalloc(arr, len(descs), stream)


def ndq_matmul_packed(format_id: int, N: int, K: int, w_ptr: int, w_len: int, x_ptr: int, M: int,
                      weight_dtype: int, out_dtype: int, y_ptr: int, stream: int = 0) -> int:
    """Raw call of the fused decode + product; returns the status code."""
    return _lib.ndq_matmul_packed(format_id, N, K, w_ptr, w_len, x_ptr, M, weight_dtype, out_dtype, y_ptr, stream)


def ndq_matmul_packed_batched(descs, K: int, x_ptr: int, M: int, weight_dtype: int, out_dtype: int,
                              stream: int = 0) -> int:
    """Raw call over a sequence of ndq_matmul_desc sharing X; returns the status code."""
    arr = (ndq_matmul_desc * max(1, len(descs)))(*descs)
    return _lib.ndq_matmul_packed_batched(arr, len(descs), K, x_ptr, M, weight_dtype, out_dtype, stream)


def ndq_test_withhold_copy(tile: int, wait_limit_us: int) -> int:
    """Raw call: the next decode launch of this host thread withholds one
    tile's staging copy (a check of the device-side failure path); returns
    the status code."""
    return _lib.ndq_test_withhold_copy(tile, wait_limit_us)


def ndq_get_device_fault() -> int:
    v = _c.c_uint32()
    rc = _lib.ndq_get_device_fault(_c.byref(v))
    if rc:
        raise NdqError(rc)
    return v.value


# ---- torch conveniences ----------------------------------------------------
def _torch():
    import torch
    return torch


def out_dtype_code(dtype) -> int:
    torch = _torch()
    return {torch.float32: NDQ_FLOAT, torch.float16: NDQ_FLOAT16, torch.bfloat16: NDQ_BFLOAT16,
            torch.float64: NDQ_DOUBLE}[dtype]


def format_id(fmt) -> int:
    if isinstance(fmt, int):
        return fmt
    i = ndq_format_from_name(fmt)
    if i < 0:
        raise NdqError(2, str(fmt))
    return i


def _stream_handle(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def dequantize_packed(fmt, shape, x, out_dtype=None, y=None, stream=None):
    """Decode one payload held in a CUDA uint8 tensor; returns y (shape `shape`)."""
    torch = _torch()
    out_dtype = out_dtype or torch.float32
    if y is None:
        y = torch.empty(tuple(int(s) for s in shape), dtype=out_dtype, device=x.device)
    if x.dtype != torch.uint8 or not x.is_contiguous() or not y.is_contiguous():
        raise ValueError("x must be a contiguous uint8 tensor and y contiguous")
    rc = ndq_dequantize_packed(format_id(fmt), shape, out_dtype_code(y.dtype), x.data_ptr(), x.numel(),
                               y.data_ptr(), _stream_handle(stream))
    if rc:
        raise NdqError(rc, str(fmt))
    return y


def make_desc(fmt, shape, x, y) -> ndq_tensor_desc:
    d = ndq_tensor_desc()
    d.format_id = format_id(fmt)
    d.ndim = len(shape)
    for i, s in enumerate(shape):
        d.shape[i] = int(s)
    d.out_dtype = out_dtype_code(y.dtype)
    d.reserved = 0
    d.x = x.data_ptr()
    d.x_len = x.numel()
    d.y = y.data_ptr()
    return d


def dequantize_packed_batched(items, workspace=None, stream=None):
    """Decode many payloads in one launch.

    items: sequence of (fmt, shape, x_uint8_cuda, y_cuda) tuples.  The
    workspace (a CUDA uint8 tensor of ndq_batched_workspace_bytes(n) bytes)
    is allocated when not given; keep it alive until the stream passes.
    Returns the workspace tensor.
    """
    torch = _torch()
    descs = [make_desc(f, s, x, y) for (f, s, x, y) in items]
    nbytes = ndq_batched_workspace_bytes(len(descs))
    if workspace is None:
        dev = items[0][2].device if items else torch.device("cuda")
        workspace = torch.empty(max(16, nbytes), dtype=torch.uint8, device=dev)
    rc = ndq_dequantize_packed_batched(descs, workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if rc:
        raise NdqError(rc)
    return workspace


def matmul_packed(fmt, w, N: int, K: int, x, out_dtype=None, y=None, stream=None, weight_dtype=None):
    """Y = X @ W^T with W [N, K] decoded from the CUDA uint8 payload `w`
    (binary32, or rounded to bfloat16 when weight_dtype is torch.bfloat16)
    and X a CUDA bfloat16 tensor [M, K]; returns Y [M, N]."""
    torch = _torch()
    out_dtype = out_dtype or torch.float32
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.shape[-1] != K:
        raise ValueError("x must be a contiguous bfloat16 tensor [M, K]")
    M = x.numel() // K if K else x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=w.device)
    wcode = out_dtype_code(weight_dtype or torch.float32)
    rc = ndq_matmul_packed(format_id(fmt), N, K, w.data_ptr(), w.numel(), x.data_ptr(), M, wcode,
                           out_dtype_code(y.dtype), y.data_ptr(), _stream_handle(stream))
    if rc:
        raise NdqError(rc, str(fmt))
    return y


def matmul_packed_batched(items, K: int, x, out_dtype=None, stream=None, weight_dtype=None):
    """Several products sharing the bfloat16 activations x [M, K]: items is
    a sequence of (fmt, w, N) or (fmt, w, N, y) with w a CUDA uint8 payload
    [N, K]; returns the list of outputs Y_i [M, N_i]."""
    torch = _torch()
    out_dtype = out_dtype or torch.float32
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.shape[-1] != K:
        raise ValueError("x must be a contiguous bfloat16 tensor [M, K]")
    M = x.numel() // K if K else x.shape[0]
    descs, ys = [], []
    for it in items:
        fmt, w, N = it[0], it[1], it[2]
        y = it[3] if len(it) > 3 and it[3] is not None else torch.empty((M, N), dtype=out_dtype, device=w.device)
        descs.append(ndq_matmul_desc(format_id(fmt), 0, N, w.data_ptr(), w.numel(), y.data_ptr()))
        ys.append(y)
    wcode = out_dtype_code(weight_dtype or torch.float32)
    odt = out_dtype_code(ys[0].dtype if ys else out_dtype)
    rc = ndq_matmul_packed_batched(descs, K, x.data_ptr(), M, wcode, odt, _stream_handle(stream))
    if rc:
        raise NdqError(rc)
    return ys


def get_device_fault() -> int:
    return ndq_get_device_fault()
