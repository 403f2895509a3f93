"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, its format table matches the pages, and host validation
(which runs before any CUDA call) agrees with the oracle's independent
length-rule implementation."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT, read_golden

import quantized_weight_block_gb300 as ndq


def _header_functions():
    text = open(os.path.join(ROOT, "include", "ndq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ndq_\w+)\s*\(", text)))


def _header_defines():
    text = open(os.path.join(ROOT, "include", "ndq.h")).read()
    return {k: int(v) for k, v in re.findall(r"#define\s+(NDQ_\w+)\s+(-?\d+)\b", text)}


def test_library_exports_every_declared_symbol():
    declared = _header_functions()
    assert len(declared) >= 10
    lib = ctypes.CDLL(ndq.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(ndq.EXPORTS) == declared


def test_binding_constants_match_header():
    d = _header_defines()
    assert d["NDQ_FLOAT"] == ndq.NDQ_FLOAT and d["NDQ_BFLOAT16"] == ndq.NDQ_BFLOAT16
    assert d["NDQ_FLOAT16"] == ndq.NDQ_FLOAT16 and d["NDQ_DOUBLE"] == ndq.NDQ_DOUBLE
    assert d["NDQ_MAX_RANK"] == ndq.NDQ_MAX_RANK and d["NDQ_NUM_FORMATS"] == ndq.NDQ_NUM_FORMATS
    for code, name in ndq.STATUS.items():
        assert d[name] == code
    # format-id macros follow the identifier table order
    for i in range(ndq.NDQ_NUM_FORMATS):
        nm = ndq.ndq_format_name(i)
        macro = "NDQ_" + nm.replace("gguf:", "GGUF_").upper()
        assert d[macro] == i, nm


def test_format_table_matches_onnx_table():
    rows = read_golden("gguf_block_table.txt")
    for i, (ident, B, S) in enumerate(rows):
        assert ndq.ndq_format_from_name(ident) == i
        assert ndq.ndq_format_name(i) == ident
        assert ndq.ndq_format_geometry(i) == (int(B), int(S))
    assert ndq.ndq_format_geometry(ndq.format_id("nvfp4")) == (64, 36)
    assert ndq.ndq_format_geometry(ndq.format_id("q4_g64_fp16")) == (64, 34)
    assert ndq.ndq_format_geometry(ndq.format_id("q8_g32_fp16")) == (32, 34)


def test_ninfer_geometry_matches_oracle(orc):
    for i in range(27, ndq.NDQ_NUM_FORMATS):
        name = ndq.ndq_format_name(i)
        assert ndq.ndq_format_geometry(i) == orc.format_info(name)[:2], name


def test_identifiers_are_closed_and_case_sensitive():
    for bad in ("gguf:Q4_0", "q4_0", "gguf:q4_0 ", "gguf:q4_0(32)", "", "NVFP4"):
        assert ndq.ndq_format_from_name(bad) == -1
    assert ndq.ndq_format_from_name(None) == -1
    n = ndq.NDQ_NUM_FORMATS
    assert ndq.ndq_format_name(-1) is None and ndq.ndq_format_name(n) is None
    with pytest.raises(ndq.NdqError):
        ndq.ndq_format_geometry(n)


def test_supported_set(orc):
    # every format the GPU decodes has an oracle decoder to be checked against
    sup = {ndq.ndq_format_name(i) for i in range(ndq.NDQ_NUM_FORMATS) if ndq.ndq_format_supported(i) == 1}
    decoded = {f for f in orc.formats() if orc.format_info(f)[2]}
    # every format the library registers is decoded by it and by the oracle
    registered = {ndq.ndq_format_name(i) for i in range(ndq.NDQ_NUM_FORMATS)}
    assert sup == registered and sup <= decoded == set(orc.formats())
    assert ndq.ndq_format_supported(99) == -1


SHAPES = [(1, 4096), (3, 7, 512), (0, 256), (5, 0), (256,), (2, 100), (-1, 256), (2**40, 2**40, 256)]


@pytest.mark.parametrize("fmt", ["gguf:q8_0", "gguf:q4_k", "gguf:mxfp4", "nvfp4", "q4_g64_fp16", "gguf:q2_k"])
@pytest.mark.parametrize("shape", SHAPES)
def test_geometry_agrees_with_oracle(orc, fmt, shape):
    B, S, _ = orc.format_info(fmt)
    cands = set()
    if all(s >= 0 for s in shape) and shape[-1] % B == 0 and max(shape) < 2**30:
        nb = int(np.prod(shape[:-1], dtype=np.int64)) * (shape[-1] // B)
        cands |= {nb * S, nb * S + 1, max(0, nb * S - 1), nb * S + 4, nb * S + 8}
    else:
        cands |= {0, 18}
    for x_len in sorted(cands):
        try:
            want = orc.geometry(fmt, shape, x_len)
            want_err = None
        except orc.OracleError as e:
            want, want_err = None, e.name
        try:
            nb, ne, nd = ndq.ndq_payload_geometry(ndq.format_id(fmt), shape, x_len)
            got_err = None
        except ndq.NdqError as e:
            got_err = e.name
        if want_err is None:
            assert got_err is None, (fmt, shape, x_len, got_err)
            assert (nb, nd) == (want[0], want[2])
            assert ne == int(np.prod(shape, dtype=np.int64))
        else:
            assert got_err == "NDQ_ERR_" + want_err.upper(), (fmt, shape, x_len, got_err, want_err)


def test_validation_errors_return_before_any_launch():
    q40 = ndq.format_id("gguf:q4_0")
    F = ndq.NDQ_FLOAT
    # invalid arguments never reach CUDA, so these run without a GPU
    assert ndq.ndq_dequantize_packed(99, (1, 32), F, 16, 18, 16) == 2
    assert ndq.ndq_dequantize_packed(q40, (), F, 16, 0, 16) == 4
    assert ndq.ndq_dequantize_packed(q40, (1,) * 9 + (32,), F, 16, 18, 16) == 4
    assert ndq.ndq_dequantize_packed(q40, (-2, 32), F, 16, 0, 16) == 5
    assert ndq.ndq_dequantize_packed(q40, (1, 33), F, 16, 18, 16) == 6
    assert ndq.ndq_dequantize_packed(q40, (1, 32), F, 16, 17, 16) == 7
    assert ndq.ndq_dequantize_packed(q40, (2**62, 2**62, 32), F, 16, 0, 16) == 8
    assert ndq.ndq_dequantize_packed(q40, (1, 32), 7, 16, 18, 16) == 9
    assert ndq.ndq_dequantize_packed(q40, (1, 32), F, 0, 18, 16) == 1
    assert ndq.ndq_dequantize_packed(q40, (1, 32), F, 16, 18, 0) == 1
    # empty tensors succeed without touching the device
    assert ndq.ndq_dequantize_packed(q40, (0, 32), F, 0, 0, 0) == 0
    assert ndq.ndq_dequantize_packed(q40, (4, 0), ndq.NDQ_BFLOAT16, 0, 0, 0) == 0


def test_batched_validation():
    q40 = ndq.format_id("gguf:q4_0")

    def desc(fmt, shape, x_len, x=16, y=16, out=ndq.NDQ_FLOAT):
        d = ndq.ndq_tensor_desc()
        d.format_id, d.ndim, d.out_dtype = fmt, len(shape), out
        for i, s in enumerate(shape):
            d.shape[i] = s
        d.x, d.x_len, d.y = x, x_len, y
        return d

    assert ndq.ndq_batched_workspace_bytes(-1) == 0
    assert ndq.ndq_batched_workspace_bytes(0) == 0
    assert ndq.ndq_batched_workspace_bytes(3) == 192
    assert ndq.ndq_dequantize_packed_batched([], 0, 0) == 0
    assert ndq._lib.ndq_dequantize_packed_batched(None, -1, None, 0, None) == 13
    good, bad = desc(q40, (1, 32), 18), desc(q40, (1, 32), 19)
    assert ndq.ndq_dequantize_packed_batched([good, bad], 16, 1 << 20) == 7  # one bad entry rejects all
    assert ndq.ndq_dequantize_packed_batched([good], 0, 1 << 20) == 10     # missing workspace
    assert ndq.ndq_dequantize_packed_batched([good], 16, 8) == 10           # too small
    assert ndq.ndq_dequantize_packed_batched([good], 24, 1 << 20) == 10     # not 16-byte aligned
    assert ndq.ndq_dequantize_packed_batched([desc(q40, (0, 32), 0, 0, 0)], 0, 0) == 0  # all empty


def test_batched_matmul_validation():
    # every product of a batched fused call is checked before any launch, so
    # these run without a GPU (one invalid descriptor rejects the call)
    q4k = ndq.format_id("gguf:q4_k")
    F, BF = ndq.NDQ_FLOAT, ndq.NDQ_BFLOAT16

    def desc(fmt, n, w_len, w=16, y=16):
        return ndq.ndq_matmul_desc(fmt, 0, n, w, w_len, y)

    K = 512
    row = K // 256 * 144
    good = desc(q4k, 3, 3 * row)
    assert ndq.ndq_matmul_packed_batched([], K, 16, 1, F, F) == 0
    assert ndq._lib.ndq_matmul_packed_batched(None, -1, K, None, 1, F, F, None) == 13
    assert ndq._lib.ndq_matmul_packed_batched(None, 2, K, None, 1, F, F, None) == 1
    assert ndq.ndq_matmul_packed_batched([good, desc(99, 3, 3 * row)], K, 16, 1, F, F) == 2
    assert ndq.ndq_matmul_packed_batched([good, desc(q4k, -1, 0)], K, 16, 1, F, F) == 5
    assert ndq.ndq_matmul_packed_batched([good], K + 32, 16, 1, F, F) == 6     # K not a multiple of 256
    assert ndq.ndq_matmul_packed_batched([good, desc(q4k, 3, 3 * row + 1)], K, 16, 1, F, F) == 7
    assert ndq.ndq_matmul_packed_batched([good, desc(q4k, 3, 3 * row, y=0)], K, 16, 1, F, F) == 1
    assert ndq.ndq_matmul_packed_batched([good], K, 0, 1, F, F) == 1           # no activations
    assert ndq.ndq_matmul_packed_batched([good], K, 16, -1, F, F) == 5
    assert ndq.ndq_matmul_packed_batched([good], K, 16, 1, 7, F) == 9          # weight type
    assert ndq.ndq_matmul_packed_batched([good], K, 16, 1, F, 10) == 9         # output type
    assert ndq.ndq_matmul_packed_batched([good], K, 16, 1, BF, ndq.NDQ_DOUBLE) == 9
    fp8 = ndq.format_id("fp8_e4m3fn_row_bf16")
    assert ndq.ndq_matmul_packed_batched([desc(fp8, 2, 2 * 40 + 4)], 40, 16, 1, F, F) == 6  # fp8 rows: K % 16
    # empty products (n = 0 or M = 0) are valid and launch nothing
    assert ndq.ndq_matmul_packed_batched([desc(q4k, 0, 0, 0, 0)], K, 16, 1, F, F) == 0
    assert ndq.ndq_matmul_packed_batched([good], K, 0, 0, F, F) == 0


def test_status_strings():
    for code in ndq.STATUS:
        assert ndq.ndq_status_string(code)
    assert ndq.ndq_status_string(1234) == "unknown status"


def test_failure_path_request_validation():
    # ndq_test_withhold_copy only records a request for the next launch of
    # this thread; out-of-range arguments are rejected
    assert ndq.ndq_test_withhold_copy(-2, 1000) == 13  # NDQ_ERR_BAD_COUNT
    assert ndq.ndq_test_withhold_copy(0, 0) == 13
    assert ndq.ndq_test_withhold_copy(0, 2000001) == 13
    assert ndq.ndq_test_withhold_copy(3, 1000) == 0
    assert ndq.ndq_test_withhold_copy(-1, 1) == 0  # cancelled
