"""CPU oracle for packed quantized-weight decoding -- TEST INFRASTRUCTURE ONLY.

A thin ctypes wrapper around ``ndq_oracle.c``: a plain, single-threaded C
decoder written from the published definitions (ONNX "DequantizePacked
decoding specification"; NInfer "tensor-formats" sections 3.3 and 4-7.2;
gld-kiln "Quantization").  It is the parity reference for the CUDA library
and the timed CPU baseline.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import it; the product library never does.
It shares no code with the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# NDQ_ORACLE_SRC / NDQ_ORACLE_LIB point the oracle at another source and
# library path; only the mutation tests use them, to check that the pins
# fail on oracles with planted mistakes.
_SRC = os.environ.get("NDQ_ORACLE_SRC") or os.path.join(_HERE, "ndq_oracle.c")
_LIB_PATH = os.environ.get("NDQ_ORACLE_LIB") or os.path.join(_HERE, "_build", "liboracle.so")
# The IQ codebooks are page data kept as a cited text fixture; the oracle
# expands them itself (oracle_set_codebook).
CODEBOOKS_FILE = os.path.join(os.path.dirname(_HERE), "tests", "golden", "iq_codebooks.txt")

# The oracle's own output-type codes (FLOAT, FLOAT16, BFLOAT16, DOUBLE).
OUT_DTYPES = {"float32": 0, "float16": 1, "bfloat16": 2, "float64": 3}
_NP_OUT = {"float32": np.float32, "float16": np.uint16, "bfloat16": np.uint16, "float64": np.float64}

ERRORS = {
    0: "ok", 1: "null", 2: "unknown_format", 3: "unsupported_format", 4: "bad_rank",
    5: "negative_dim", 6: "not_block_aligned", 7: "length_mismatch", 8: "overflow",
    9: "bad_dtype", 10: "range", 11: "encode",
}


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        self.name = ERRORS.get(code, str(code))
        super().__init__(f"oracle error {self.name} ({code}) {what}")


def build(force: bool = False) -> str:
    """Compile the oracle with strict binary32 rounding (no FP contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        c = ctypes
        i64p, u8p, vp = c.POINTER(c.c_int64), c.POINTER(c.c_uint8), c.c_void_p
        L.oracle_format_count.restype = c.c_int
        L.oracle_format_name.restype = c.c_char_p
        L.oracle_format_name.argtypes = [c.c_int]
        L.oracle_format_info.argtypes = [c.c_char_p, c.POINTER(c.c_int), c.POINTER(c.c_int), c.POINTER(c.c_int)]
        L.oracle_geometry.argtypes = [c.c_char_p, i64p, c.c_int, c.c_uint64, c.POINTER(c.c_uint64),
                                      c.POINTER(c.c_uint64), c.POINTER(c.c_uint64)]
        L.oracle_decode.argtypes = [c.c_char_p, i64p, c.c_int, c.c_int, vp, c.c_uint64, vp]
        L.oracle_decode_range.argtypes = [c.c_char_p, i64p, c.c_int, c.c_int, vp, c.c_uint64,
                                          c.c_uint64, c.c_uint64, vp]
        L.oracle_decode_block_f32.argtypes = [c.c_char_p, vp, c.c_float, vp]
        L.oracle_h2f.restype = c.c_float
        L.oracle_h2f.argtypes = [c.c_uint16]
        for fn in ("oracle_e8m0_half", "oracle_ue4m3_half", "oracle_e4m3fn", "oracle_e2m1"):
            getattr(L, fn).restype = c.c_float
            getattr(L, fn).argtypes = [c.c_uint8]
        for fn in ("oracle_f32_to_bf16", "oracle_f32_to_f16"):
            getattr(L, fn).restype = c.c_uint16
            getattr(L, fn).argtypes = [c.c_uint32]
        L.oracle_kiln_group_count.restype = c.c_uint64
        L.oracle_kiln_group_count.argtypes = [i64p, c.c_int, c.c_int, c.c_uint64]
        L.oracle_grouped_absmax_group.argtypes = [vp, c.c_int, c.c_int, c.c_int, vp, vp]
        L.oracle_encode_grouped.argtypes = [c.c_char_p, vp, c.c_uint64, c.c_uint64, vp]
        for fn in ("oracle_h2f_array", "oracle_f32_to_bf16_array", "oracle_f32_to_f16_array"):
            getattr(L, fn).argtypes = [vp, vp, c.c_uint64]
        L.oracle_matmul_packed.argtypes = [c.c_char_p, c.c_uint64, c.c_uint64, vp, c.c_uint64, vp, c.c_uint64,
                                           c.c_int, vp, vp]
        L.oracle_set_codebook.argtypes = [c.c_char_p, c.c_int, c.c_int, vp, c.c_int, vp, c.c_uint64]
        L.oracle_codebook_row.argtypes = [c.c_char_p, c.c_int, vp]
        L.oracle_codebook_rows.argtypes = [c.c_char_p]
        for name, (width, bits, _rows, values, packed) in read_codebooks().items():
            vals = np.array(values, np.int32)
            rc = L.oracle_set_codebook(name.encode(), width, bits, _ptr(vals), len(vals), _ptr(packed), packed.size)
            if rc:
                raise OracleError(rc, f"codebook {name}")
        _lib = L
    return _lib


def read_codebooks(path: str = CODEBOOKS_FILE) -> dict:
    """{name: (width, bits, stated rows, values, packed bytes)} from the fixture."""
    books, cur = {}, None
    with open(path) as f:
        for line in f:
            tok = line.split("#", 1)[0].split()
            if not tok:
                continue
            if tok[0] == "codebook":
                cur = tok[1]
                books[cur] = [int(tok[2]), int(tok[3]), int(tok[4]), [int(v) for v in tok[5].split(",")], []]
            elif tok[0] == "hex":
                books[cur][4].append(tok[1])
    return {k: (w, b, r, v, np.frombuffer(bytes.fromhex("".join(h)), np.uint8).copy())
            for k, (w, b, r, v, h) in books.items()}


def matmul_packed(name: str, N: int, K: int, w: np.ndarray, x_bf16: np.ndarray, weights: str = "bfloat16"):
    """Reference of the fused decode + product: (y, yabs), both float64 [M, N].

    y[m, n] = sum_k X[m, k] * W[n, k] with W the payload decoded to
    `weights` ("float32": the exact binary32 decode, or "bfloat16") and X
    given as bfloat16 bit patterns [M, K]; yabs is sum_k |X W|."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1, K) if K else np.zeros((len(x_bf16), 0), np.uint16)
    M = x.shape[0]
    y = np.zeros((M, N), np.float64)
    yabs = np.zeros((M, N), np.float64)
    rc = lib().oracle_matmul_packed(name.encode(), N, K, _ptr(w), w.size, _ptr(x), M, OUT_DTYPES[weights],
                                    _ptr(y), _ptr(yabs))
    if rc:
        raise OracleError(rc, name)
    return y, yabs


def codebook_rows(name: str) -> int:
    return lib().oracle_codebook_rows(name.encode())


def codebook_row(name: str, r: int) -> list[int]:
    out = np.zeros(8, np.int32)
    w = lib().oracle_codebook_row(name.encode(), r, _ptr(out))
    if w < 0:
        raise OracleError(-w, f"{name} row {r}")
    return out[:w].tolist()


def _shape_arg(shape):
    arr = (ctypes.c_int64 * max(1, len(shape)))(*[int(s) for s in shape])
    return arr, len(shape)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def formats() -> list[str]:
    L = lib()
    return [L.oracle_format_name(i).decode() for i in range(L.oracle_format_count())]


def format_info(name: str) -> tuple[int, int, bool]:
    B, S, dec = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = lib().oracle_format_info(name.encode(), ctypes.byref(B), ctypes.byref(S), ctypes.byref(dec))
    if rc:
        raise OracleError(rc, name)
    return B.value, S.value, bool(dec.value)


def geometry(name: str, shape, x_len: int) -> tuple[int, int, int]:
    """(nblocks, rows, divisor count) under the length rule, or OracleError."""
    sa, nd = _shape_arg(shape)
    nb, rows, nd_ = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
    rc = lib().oracle_geometry(name.encode(), sa, nd, x_len, ctypes.byref(nb), ctypes.byref(rows), ctypes.byref(nd_))
    if rc:
        raise OracleError(rc, name)
    return nb.value, rows.value, nd_.value


def decode(name: str, shape, x: np.ndarray, out_dtype: str = "float32") -> np.ndarray:
    """Decode a whole payload. 16-bit outputs come back as uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.uint8)
    n = int(np.prod(shape, dtype=np.int64)) if len(shape) else 0
    y = np.empty(n, dtype=_NP_OUT[out_dtype])
    sa, nd = _shape_arg(shape)
    rc = lib().oracle_decode(name.encode(), sa, nd, OUT_DTYPES[out_dtype], _ptr(x), x.size, _ptr(y))
    if rc:
        raise OracleError(rc, name)
    return y.reshape(tuple(int(s) for s in shape))


def decode_range(name: str, shape, x: np.ndarray, b0: int, b1: int, out_dtype: str = "float32") -> np.ndarray:
    """Decode blocks [b0, b1) of a payload; returns (b1-b0)*B values (flat)."""
    x = np.ascontiguousarray(x, dtype=np.uint8)
    B, _, _ = format_info(name)
    y = np.empty((b1 - b0) * B, dtype=_NP_OUT[out_dtype])
    sa, nd = _shape_arg(shape)
    rc = lib().oracle_decode_range(name.encode(), sa, nd, OUT_DTYPES[out_dtype], _ptr(x), x.size, b0, b1, _ptr(y))
    if rc:
        raise OracleError(rc, name)
    return y


def decode_range_into(name: str, shape, x: np.ndarray, b0: int, b1: int, out_dtype: str, y: np.ndarray) -> None:
    """Decode blocks [b0, b1) of a payload into the contiguous array y
    ((b1-b0)*B elements of the output type; 16-bit outputs as uint16)."""
    assert y.flags.c_contiguous and y.dtype == _NP_OUT[out_dtype]
    B, _, _ = format_info(name)
    assert y.size == (b1 - b0) * B
    sa, nd = _shape_arg(shape)
    rc = lib().oracle_decode_range(name.encode(), sa, nd, OUT_DTYPES[out_dtype], _ptr(x), x.size, b0, b1, _ptr(y))
    if rc:
        raise OracleError(rc, name)


def decode_parallel(name: str, shape, x: np.ndarray, out_dtype: str = "float32", threads: int | None = None,
                    pool=None) -> np.ndarray:
    """The same result as decode(), with the block range split into disjoint
    pieces decoded by host threads (each piece by the unchanged
    single-threaded C decoder; ctypes releases the GIL during the call)."""
    import concurrent.futures as cf

    x = np.ascontiguousarray(x, dtype=np.uint8)
    nb, _, _ = geometry(name, shape, x.size)
    B, _, _ = format_info(name)
    y = np.empty(nb * B, dtype=_NP_OUT[out_dtype])
    threads = threads or os.cpu_count() or 1
    step = max(1, -(-nb // (4 * threads)))
    ranges = [(b0, min(nb, b0 + step)) for b0 in range(0, nb, step)]

    def run(r):
        decode_range_into(name, shape, x, r[0], r[1], out_dtype, y[r[0] * B:r[1] * B])

    if pool is not None:
        list(pool.map(run, ranges))
    else:
        with cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, ranges))
    return y.reshape(tuple(int(s) for s in shape))


def decode_block_f32(name: str, block: bytes | np.ndarray, dw: float = 1.0) -> np.ndarray:
    """One block to binary32 values (no cast)."""
    B, S, _ = format_info(name)
    b = np.frombuffer(bytes(block), dtype=np.uint8)
    if b.size != S:
        raise ValueError(f"{name} block must be {S} bytes, got {b.size}")
    y = np.empty(B, dtype=np.float32)
    rc = lib().oracle_decode_block_f32(name.encode(), _ptr(np.ascontiguousarray(b)), ctypes.c_float(dw), _ptr(y))
    if rc:
        raise OracleError(rc, name)
    return y


def h2f(u16) -> np.ndarray:
    a = np.ascontiguousarray(u16, dtype=np.uint16)
    out = np.empty(a.size, dtype=np.float32)
    lib().oracle_h2f_array(_ptr(a), _ptr(out), a.size)
    return out


def f32_to_bf16(bits_u32) -> np.ndarray:
    a = np.ascontiguousarray(bits_u32, dtype=np.uint32)
    out = np.empty(a.size, dtype=np.uint16)
    lib().oracle_f32_to_bf16_array(_ptr(a), _ptr(out), a.size)
    return out


def f32_to_f16(bits_u32) -> np.ndarray:
    a = np.ascontiguousarray(bits_u32, dtype=np.uint32)
    out = np.empty(a.size, dtype=np.uint16)
    lib().oracle_f32_to_f16_array(_ptr(a), _ptr(out), a.size)
    return out


def e8m0_half(e: int) -> float:
    return lib().oracle_e8m0_half(e)


def ue4m3_half(e: int) -> float:
    return lib().oracle_ue4m3_half(e)


def e4m3fn(w: int) -> float:
    return lib().oracle_e4m3fn(w)


def e2m1(c: int) -> float:
    return lib().oracle_e2m1(c)


def kiln_group_count(shape, axis: int, g: int) -> int:
    sa, nd = _shape_arg(shape)
    return lib().oracle_kiln_group_count(sa, nd, axis, g)


def grouped_absmax_group(x, qmin: int, qmax: int) -> tuple[int, np.ndarray]:
    """grouped_absmax on one group: (binary16 scale bits, integer codes)."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    s = np.zeros(1, dtype=np.uint16)
    codes = np.zeros(a.size, dtype=np.int32)
    rc = lib().oracle_grouped_absmax_group(_ptr(a), a.size, qmin, qmax, _ptr(s), _ptr(codes))
    if rc:
        raise OracleError(rc, "grouped_absmax")
    return int(s[0]), codes


def encode_grouped(name: str, x: np.ndarray) -> np.ndarray:
    """Encode a [rows, K] float32 matrix into a q4/q5/q6_g64_fp16 or
    q8_g32_fp16 payload (grouped_absmax, NInfer section 7.2)."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    rows, K = a.shape
    G, S, _ = format_info(name)
    out = np.zeros(rows * (K // G) * S, dtype=np.uint8)
    rc = lib().oracle_encode_grouped(name.encode(), _ptr(a), rows, K, _ptr(out))
    if rc:
        raise OracleError(rc, name)
    return out
