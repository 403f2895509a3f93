"""GPU test of ndq_dequantize_packed_batched_noalloc.

That entry point serves callers that cannot allocate device memory (for
example a C or plugin host whose device memory belongs to another
framework's pool): it keeps the batched launch table in a fixed array inside
the library instead of a caller-provided workspace.  Here it is called
through the C ABI and must reproduce, bit for bit (NaN only needs to be
NaN), what the workspace-based ndq_dequantize_packed_batched produces on the
same batch, and what the CPU oracle decodes, on two calls in a row with
different batches (so the second call has to overwrite the table the first
one left behind).  One pair of calls uses more than 128 tensors, so the
table is written by several upload launches, the second call shorter than
the first.  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_bit_exact

pytestmark = pytest.mark.gpu

import quantized_weight_block_gb300 as ndq  # noqa: E402

TORCH_OUT = {"float32": torch.float32, "float16": torch.float16, "bfloat16": torch.bfloat16,
             "float64": torch.float64}
FORMATS = ["gguf:q8_0", "q8_g32_fp16", "gguf:q4_0", "gguf:iq4_nl", "gguf:q4_k", "gguf:q6_k",
           "gguf:mxfp4", "gguf:nvfp4", "nvfp4", "q4_g64_fp16"]


def _batch(seed: int):
    rng = np.random.default_rng(seed)
    specs = []
    for i, fmt in enumerate(FORMATS):
        B, _ = synth.GEOMETRY[fmt]
        shape = (int(rng.integers(1, 6)), int(rng.integers(1, 70)) * B)
        out = list(TORCH_OUT)[(i + seed) % 4]
        specs.append((fmt, shape, out, synth.payload(fmt, shape, seed=seed * 100 + i, dist="bytes")))
    return specs


def _many_small(n: int, seed: int):
    # n tensors of one or two blocks each, formats and output types mixed
    rng = np.random.default_rng(seed)
    specs = []
    for i in range(n):
        fmt = FORMATS[int(rng.integers(0, len(FORMATS)))]
        B, _ = synth.GEOMETRY[fmt]
        shape = (1, B * int(rng.integers(1, 3)))
        out = list(TORCH_OUT)[int(rng.integers(0, 4))]
        specs.append((fmt, shape, out, synth.payload(fmt, shape, seed=seed * 1000 + i, dist="bytes")))
    return specs


def _descs(specs):
    descs, ys, keep = [], [], []
    for fmt, shape, out, x in specs:
        xt = torch.from_numpy(x).cuda()
        y = torch.full(shape, float("nan"), dtype=TORCH_OUT[out], device="cuda")
        descs.append(ndq.make_desc(fmt, shape, xt, y))
        ys.append(y)
        keep.append(xt)
    return descs, ys, keep


def _bits(y, out):
    return y.cpu().view(torch.uint16 if out in ("float16", "bfloat16") else TORCH_OUT[out]).numpy()


def _with_workspace(specs):
    descs, ys, keep = _descs(specs)
    ws_bytes = ndq.ndq_batched_workspace_bytes(len(descs))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    rc = ndq.ndq_dequantize_packed_batched(descs, ws.data_ptr(), ws_bytes, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ndq.ndq_status_string(rc)
    torch.cuda.synchronize()
    return [_bits(y, s[2]) for y, s in zip(ys, specs)]


def _two_calls_in_a_row(orc, batches):
    expected = [_with_workspace(b) for b in batches]
    stream = torch.cuda.current_stream().cuda_stream
    runs = []
    for b in batches:  # calls in a row on the same stream
        descs, ys, keep = _descs(b)
        rc = ndq.ndq_dequantize_packed_batched_noalloc(descs, stream)
        assert rc == 0, ndq.ndq_status_string(rc)
        runs.append((ys, keep))
    torch.cuda.synchronize()
    for b, exp, (ys, _) in zip(batches, expected, runs):
        for (fmt, shape, out, x), want, y in zip(b, exp, ys):
            got = _bits(y, out)
            assert_bit_exact(got, want, out, f"no-alloc vs workspace call {fmt} {shape} {out}")
            assert_bit_exact(got, orc.decode(fmt, shape, x, out), out, f"no-alloc vs oracle {fmt} {shape} {out}")
    assert ndq.get_device_fault() == 0


def test_noalloc_matches_workspace_call_and_oracle_on_two_calls(orc):
    _two_calls_in_a_row(orc, [_batch(1), _batch(2)])


def test_noalloc_tables_of_several_upload_chunks(orc):
    # 300 tensors (three upload launches), then 150 (two): the second call
    # rewrites the first 150 entries and leaves the rest of the first table
    _two_calls_in_a_row(orc, [_many_small(300, 3), _many_small(150, 4)])


def test_noalloc_rejects_batches_beyond_its_table():
    d = ndq.ndq_tensor_desc()
    descs = [d] * (ndq.NDQ_NOALLOC_MAX_TENSORS + 1)
    assert ndq.ndq_dequantize_packed_batched_noalloc(descs, 0) == 14  # NDQ_ERR_TOO_MANY_TENSORS
    assert ndq.ndq_dequantize_packed_batched_noalloc([], 0) == 0
