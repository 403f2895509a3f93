"""GPU parity: the CUDA decode (through the C ABI) against the CPU oracle,
bit for bit (0 ULP in FP32 and after the single RNE cast; NaN only needs to
be NaN), on seeded synthetic payloads.  Sizes span several 8192-element
tiles with a ragged last tile; edge cases cover unaligned payload/output
pointers, empty tensors, rank 1 and rank 3, several nvfp4 divisors, every
special scale byte, and batched launches mixing formats and output types."""
import zlib

import numpy as np
import pytest
import torch

import synth
from conftest import assert_bit_exact

pytestmark = pytest.mark.gpu

import quantized_weight_block_gb300 as ndq  # noqa: E402

FORMATS = ["gguf:q8_0", "q8_g32_fp16", "gguf:q4_0", "gguf:iq4_nl", "gguf:q4_k", "gguf:q6_k",
           "gguf:mxfp4", "gguf:nvfp4", "nvfp4", "q4_g64_fp16"] + synth.NEXT_FORMATS
OUTS = ["float32", "float16", "bfloat16", "float64"]
TORCH_OUT = {"float32": torch.float32, "float16": torch.float16, "bfloat16": torch.bfloat16,
             "float64": torch.float64}
DEV = "cuda"


def ragged_shape(fmt, rows=3):
    B, _ = synth.GEOMETRY[fmt]
    # about 11.7 tiles of 8192 elements in total over `rows` rows, not a multiple of a tile
    per_row = (8192 * 11 + 5 * 8192 // 7) // rows // B * B
    return (rows, per_row)


def gpu_decode(fmt, shape, x_np, out, x_offset=0, y_offset=0):
    """Decode through the C ABI; offsets (bytes / elements) misalign x / y."""
    xs = torch.zeros(x_np.size + x_offset + 16, dtype=torch.uint8, device=DEV)
    xs[x_offset:x_offset + x_np.size] = torch.from_numpy(x_np).to(DEV)
    x = xs[x_offset:x_offset + x_np.size]
    n = int(np.prod(shape, dtype=np.int64))
    ybuf = torch.full((n + y_offset + 8,), float("nan"), dtype=TORCH_OUT[out], device=DEV)
    y = ybuf[y_offset:y_offset + n]
    rc = ndq.ndq_dequantize_packed(ndq.format_id(fmt), shape, ndq.out_dtype_code(TORCH_OUT[out]),
                                   x.data_ptr(), x_np.size, y.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ndq.ndq_status_string(rc)
    torch.cuda.synchronize()
    # guard elements around y are untouched
    if y_offset:
        assert torch.isnan(ybuf[:y_offset].float()).all()
    assert torch.isnan(ybuf[y_offset + n:].float()).all()
    return y.cpu().view(torch.uint16 if out in ("float16", "bfloat16") else TORCH_OUT[out]).numpy()


@pytest.fixture(autouse=True)
def _no_device_fault():
    yield
    assert ndq.get_device_fault() == 0


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("out", OUTS)
@pytest.mark.parametrize("dist", ["workload", "bytes"])
def test_parity_ragged(orc, fmt, out, dist):
    shape = ragged_shape(fmt)
    x = synth.payload(fmt, shape, seed=zlib.crc32(f"{fmt}/{dist}".encode()) % 1000, dist=dist)
    want = orc.decode(fmt, shape, x, out)
    got = gpu_decode(fmt, shape, x, out)
    assert_bit_exact(got, want, out, f"{fmt} {out} {dist}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("x_off,y_off", [(1, 0), (3, 1), (8, 3), (0, 1), (5, 4)])
def test_parity_unaligned_pointers(orc, fmt, x_off, y_off):
    shape = ragged_shape(fmt, rows=2)
    x = synth.payload(fmt, shape, seed=17, dist="bytes")
    for out in ("bfloat16", "float32"):
        want = orc.decode(fmt, shape, x, out)
        got = gpu_decode(fmt, shape, x, out, x_offset=x_off, y_offset=y_off)
        assert_bit_exact(got, want, out, f"{fmt} {out} x+{x_off} y+{y_off}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_parity_small_and_odd_shapes(orc, fmt):
    B, _ = synth.GEOMETRY[fmt]
    for shape in [(B,), (1, B), (2, 3, 2 * B), (1, 8192 // B * B), (1, 8192 + B), (5, 3 * B), (8192 // B + 1, B)]:
        if fmt == "nvfp4" and len(shape) == 1:
            shape = (1, B)
        x = synth.payload(fmt, shape, seed=3, dist="bytes")
        for out in ("float32", "bfloat16"):
            assert_bit_exact(gpu_decode(fmt, shape, x, out), orc.decode(fmt, shape, x, out), out, f"{fmt} {shape}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_empty_tensors(fmt):
    B, _ = synth.GEOMETRY[fmt]
    for shape in [(0, B), (4, 0), (0,)]:
        y = torch.empty(0, dtype=torch.bfloat16, device=DEV)
        rc = ndq.ndq_dequantize_packed(ndq.format_id(fmt), shape, ndq.NDQ_BFLOAT16, 0, 0, y.data_ptr() or 0, 0)
        assert rc == 0


@pytest.mark.parametrize("ndiv,rows", [(1, 6), (2, 6), (3, 6), (6, 6), (7, 21), (5, 640)])
def test_nvfp4_divisors(orc, ndiv, rows):
    shape = (rows, 64 * 45)  # 45 blocks per row: tiles straddle rows and divisors
    x = synth.payload("nvfp4", shape, seed=ndiv, dist="workload", ndiv=ndiv)
    for out in ("float32", "bfloat16"):
        assert_bit_exact(gpu_decode("nvfp4", shape, x, out), orc.decode("nvfp4", shape, x, out), out,
                         f"nvfp4 D={ndiv}")


def test_nvfp4_every_scale_code_pair(orc):
    # 256 scale bytes x 16 codes, divisors that exercise rounding
    codes = np.array([(c | ((15 - c) << 4)) for c in range(8)] * 4, np.uint8)  # all 16 codes per group
    blocks = []
    for s in range(256):
        blocks.append(np.concatenate([np.full(4, s, np.uint8), codes]))
    blk = np.concatenate(blocks)
    for dw in (1.0, 26880.0, 3.0, 1e-30, 3e38, -0.75):
        x = np.concatenate([blk, np.array([dw], "<f4").view(np.uint8)])
        for out in ("float32", "bfloat16", "float16"):
            assert_bit_exact(gpu_decode("nvfp4", (256, 64), x, out), orc.decode("nvfp4", (256, 64), x, out),
                             out, f"dw={dw}")


@pytest.mark.parametrize("fmt", ["gguf:mxfp4", "gguf:nvfp4"])
def test_every_scale_byte(orc, fmt):
    B, S = synth.GEOMETRY[fmt]
    nsc = 1 if fmt == "gguf:mxfp4" else 4
    codes = np.array([(c | ((15 - c) << 4)) for c in range(8)] * ((S - nsc) // 8), np.uint8)
    x = np.concatenate([np.concatenate([np.full(nsc, s, np.uint8), codes]) for s in range(256)])
    for out in OUTS:
        assert_bit_exact(gpu_decode(fmt, (256, B), x, out), orc.decode(fmt, (256, B), x, out), out, fmt)


def test_special_binary16_scales(orc):
    # every binary16 scale pattern class: zeros, subnormals, max, inf, NaN,
    # placed in the first (d) and second (m / dmin) binary16 field
    specials = np.array([0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00, 0x7E00, 0x7C01,
                         0x3C00, 0xBC00], np.uint16)
    fields = {"gguf:q8_0": (0,), "gguf:q4_0": (0,), "gguf:iq4_nl": (0,), "q4_g64_fp16": (0,), "gguf:q4_k": (0, 2),
              "gguf:q6_k": (208,), **synth.F16_SCALES, "q2_g64_fp16": (0,), "q5_g64_fp16": (0,), "q6_g64_fp16": (0,),
              "t2_g128_fp16": (0,)}
    for fmt, offs in fields.items():
        B, S = synth.GEOMETRY[fmt]
        nb = len(specials) ** 2
        x = synth.payload(fmt, (nb, B), seed=5, dist="bytes").reshape(nb, S).copy()
        a, b = np.meshgrid(specials, specials)
        x[:, offs[0]:offs[0] + 2] = a.reshape(-1, 1).view(np.uint8).reshape(nb, 2)
        if len(offs) > 1:
            x[:, offs[1]:offs[1] + 2] = b.reshape(-1, 1).view(np.uint8).reshape(nb, 2)
        x = x.reshape(-1)
        for out in OUTS:
            assert_bit_exact(gpu_decode(fmt, (nb, B), x, out), orc.decode(fmt, (nb, B), x, out), out, fmt)


def test_special_binary32_scales_q8_k(orc):
    # gguf:q8_k's scale is binary32: zeros, subnormals, max, inf, NaN
    specials = np.array([0, 0x80000000, 1, 0x807FFFFF, 0x00800000, 0x7F7FFFFF, 0xFF7FFFFF, 0x7F800000,
                         0xFF800000, 0x7FC00000, 0x7F800001, 0x3F800000, 0x477FE000, 0x5F800000], np.uint32)
    nb = len(specials) * 4
    x = synth.payload("gguf:q8_k", (nb, 256), seed=6, dist="bytes").reshape(nb, 292).copy()
    x[:, 0:4] = np.repeat(specials, 4).astype("<u4").view(np.uint8).reshape(nb, 4)
    x = x.reshape(-1)
    for out in OUTS:
        assert_bit_exact(gpu_decode("gguf:q8_k", (nb, 256), x, out), orc.decode("gguf:q8_k", (nb, 256), x, out), out,
                         "q8_k")


def test_special_binary16_scales_iq1_m(orc):
    # gguf:iq1_m's binary16 scale is the top nibbles of the four 16-bit words
    # at byte 48 (nibble k in word k)
    specials = [0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00, 0x7E00, 0x7C01, 0x3C00, 0xBC00]
    nb = len(specials) * 3
    x = synth.payload("gguf:iq1_m", (nb, 256), seed=7, dist="bytes").reshape(nb, 56).copy()
    for r in range(nb):
        h = specials[r % len(specials)]
        for k in range(4):
            x[r, 49 + 2 * k] = (x[r, 49 + 2 * k] & 0x0F) | (((h >> (4 * k)) & 15) << 4)
    x = x.reshape(-1)
    for out in OUTS:
        assert_bit_exact(gpu_decode("gguf:iq1_m", (nb, 256), x, out), orc.decode("gguf:iq1_m", (nb, 256), x, out),
                         out, "iq1_m")


@pytest.mark.parametrize("fmt", synth.ROW_SCALED)
def test_fp8_rows_every_code_and_special_multipliers(orc, fmt):
    # 256 codes per row (every E4M3FN word), one special multiplier per row:
    # zeros, subnormals, largest finite, infinities, NaN, negative
    words = [0x0000, 0x8000, 0x0001, 0x8001, 0x3F80, 0xBF80, 0x7F7F, 0x7F80, 0xFF80, 0x7FC0, 0x0080, 0x4B00] \
        if fmt == "fp8_e4m3fn_row_bf16" else \
        [0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0xBC00, 0x7BFF, 0x7C00, 0xFC00, 0x7E00, 0x5A00]
    N = len(words)
    x = np.concatenate([np.tile(np.arange(256, dtype=np.uint8), N), np.array(words, "<u2").view(np.uint8)])
    for out in OUTS:
        assert_bit_exact(gpu_decode(fmt, (N, 256), x, out), orc.decode(fmt, (N, 256), x, out), out, fmt)


@pytest.mark.parametrize("fmt", synth.ROW_SCALED)
@pytest.mark.parametrize("shape", [(7, 1), (3, 5), (2, 15), (4, 16), (3, 17), (1, 8191), (2, 8193), (1000, 13),
                                   (9, 4097), (2, 3, 11), (37,)])
def test_fp8_rows_cross_units_and_tiles(orc, fmt, shape):
    # rows that are not a multiple of 16 codes: 16-code units straddle rows,
    # and a partial last unit
    x = synth.payload(fmt, shape, seed=sum(shape), dist="workload")
    for out in ("float32", "bfloat16"):
        for x_off, y_off in ((0, 0), (3, 1)):
            assert_bit_exact(gpu_decode(fmt, shape, x, out, x_offset=x_off, y_offset=y_off),
                             orc.decode(fmt, shape, x, out), out, f"{fmt} {shape} x+{x_off} y+{y_off}")


def test_batched_mixed(orc):
    specs = []
    rng = np.random.default_rng(0)
    for i, fmt in enumerate(FORMATS * 2):
        B, _ = synth.GEOMETRY[fmt]
        rows = int(rng.integers(1, 9))
        k = int(rng.integers(1, 40)) * B
        out = OUTS[i % 4]
        specs.append((fmt, (rows, k), out, synth.payload(fmt, (rows, k), seed=200 + i, dist="bytes")))
    specs.insert(3, ("gguf:q4_k", (0, 256), "bfloat16", np.zeros(0, np.uint8)))  # empty entry
    items, ys = [], []
    for fmt, shape, out, x in specs:
        xt = torch.from_numpy(x).to(DEV) if x.size else torch.empty(0, dtype=torch.uint8, device=DEV)
        y = torch.empty(shape, dtype=TORCH_OUT[out], device=DEV)
        items.append((fmt, shape, xt, y))
        ys.append(y)
    ws = ndq.dequantize_packed_batched(items)
    torch.cuda.synchronize()
    del ws
    for (fmt, shape, out, x), y in zip(specs, ys):
        if not x.size:
            continue
        got = y.cpu().view(torch.uint16 if out in ("float16", "bfloat16") else TORCH_OUT[out]).numpy()
        assert_bit_exact(got, orc.decode(fmt, shape, x, out), out, f"batched {fmt} {out}")


def test_batched_nvfp4_divisors(orc):
    # one launch of nvfp4 tensors to a 16-bit output (the byte-table kernel):
    # the table serves the first tensor's divisor, tensors with another
    # divisor (or several) divide per element, and a tensor whose divisor
    # equals the first one's uses the table again
    specs = []
    for i, (dw, ndiv) in enumerate(((26880.0, 1), (3.0, 1), (26880.0, 1), (0.5, 1), (None, 3))):
        shape = (3 * (i + 1), 64 * 70)
        x = synth.payload("nvfp4", shape, seed=60 + i, ndiv=ndiv).copy()
        if dw is not None:
            x[-4:] = np.array([dw], "<f4").view(np.uint8)
        specs.append((shape, x))
    for out in ("bfloat16", "float16"):
        items, ys = [], []
        for shape, x in specs:
            y = torch.empty(shape, dtype=TORCH_OUT[out], device=DEV)
            items.append(("nvfp4", shape, torch.from_numpy(x).to(DEV), y))
            ys.append(y)
        ws = ndq.dequantize_packed_batched(items)
        torch.cuda.synchronize()
        del ws
        for (shape, x), y in zip(specs, ys):
            got = y.cpu().view(torch.uint16).numpy()
            assert_bit_exact(got, orc.decode("nvfp4", shape, x, out), out, f"batched nvfp4 {shape} {out}")


def test_repeat_is_deterministic():
    fmt, shape = "gguf:q6_k", (64, 4096)
    x = torch.from_numpy(synth.payload(fmt, shape, seed=1)).to(DEV)
    a = ndq.dequantize_packed(fmt, shape, x, torch.bfloat16)
    b = ndq.dequantize_packed(fmt, shape, x, torch.bfloat16)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---- full-size workloads: every output element against the oracle -------
# The oracle decodes these with its block range split over the host cores
# (oracle.decode_parallel: the unchanged single-threaded decoder per piece).
def _bits_of(y, out):
    return y.cpu().view(torch.uint16 if out in ("float16", "bfloat16") else TORCH_OUT[out]).numpy()


@pytest.mark.parametrize("label,fmt,shape,seed,out", synth.WORKLOADS + synth.NEXT_WORKLOADS)
def test_full_size_workloads(orc, label, fmt, shape, seed, out):
    """Each single-format workload at its full size, in the launch the
    benchmark times (one ndq_dequantize_packed call), compared whole."""
    x = synth.payload(fmt, shape, seed)
    y = ndq.dequantize_packed(fmt, shape, torch.from_numpy(x).to(DEV), TORCH_OUT[out])
    torch.cuda.synchronize()
    assert_bit_exact(_bits_of(y, out), orc.decode_parallel(fmt, shape, x, out), out, label)


def _whole_model_payloads(specs):
    import concurrent.futures as cf

    with cf.ThreadPoolExecutor(8) as ex:
        return list(ex.map(lambda s: synth.payload(s.fmt, s.shape, s.seed), specs))


def test_whole_model_batched_full(orc):
    """The whole-model workload in the launch configuration the benchmark
    times (one batched launch over all 225 tensors, the q8_0 / q4_k / q6_k
    kernel), every element of every tensor compared with the oracle, one
    tensor at a time so that host memory holds one decoded tensor at most."""
    import concurrent.futures as cf

    specs = synth.llama3_8b_tensors()
    xs_np = _whole_model_payloads(specs)
    items = []
    for s, x in zip(specs, xs_np):
        items.append((s.fmt, s.shape, torch.from_numpy(x).to(DEV),
                      torch.full(s.shape, float("nan"), dtype=torch.bfloat16, device=DEV)))
    ws = ndq.dequantize_packed_batched(items)
    torch.cuda.synchronize()
    del ws
    with cf.ThreadPoolExecutor() as pool:
        for s, x, it in zip(specs, xs_np, items):
            want = orc.decode_parallel(s.fmt, s.shape, x, "bfloat16", pool=pool)
            assert_bit_exact(_bits_of(it[3], "bfloat16"), want, "bfloat16", f"whole model {s.name}")


def _batch_and_check(orc, specs, what):
    """One batched call over specs = [(fmt, shape, out, payload)], every
    output compared whole."""
    items, ys = [], []
    for fmt, shape, out, x in specs:
        y = torch.full(shape, float("nan"), dtype=TORCH_OUT[out], device=DEV)
        items.append((fmt, shape, torch.from_numpy(x).to(DEV), y))
        ys.append(y)
    ws = ndq.dequantize_packed_batched(items)
    torch.cuda.synchronize()
    del ws
    for (fmt, shape, out, x), y in zip(specs, ys):
        assert_bit_exact(_bits_of(y, out), orc.decode_parallel(fmt, shape, x, out), out, f"{what} {fmt} {shape}")


def _ring_wrapping_tiles():
    # more tiles than every resident CTA can hold in its staging ring, twice
    # over, so every CTA reuses each stage several times
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return sms * 3 * 4 * 2


@pytest.mark.parametrize("out", OUTS)
def test_batched_kquant_mix_ring_wraps(orc, out):
    """A batch of only gguf:q8_0 / q4_k / q6_k tensors (the whole-model
    kernel) of one output type, large enough that the staging ring of every
    CTA wraps several times, with ragged row counts; compared whole."""
    tiles = _ring_wrapping_tiles()
    rng = np.random.default_rng(11)
    specs, n = [], 0
    i = 0
    while n < tiles * 8192:
        fmt = ("gguf:q8_0", "gguf:q4_k", "gguf:q6_k")[i % 3]
        shape = (int(rng.integers(50, 700)), int(rng.choice([1024, 4096, 2816])))
        specs.append((fmt, shape, out, synth.payload(fmt, shape, seed=300 + i)))
        n += shape[0] * shape[1]
        i += 1
    _batch_and_check(orc, specs, f"k-quant mix {out}")


@pytest.mark.parametrize("outs", [["bfloat16"], OUTS])
def test_batched_all_formats_ring_wraps(orc, outs):
    """Every format in one batched launch (one output type: the all-format
    kernel of that type; mixed types: the generic kernel), each CTA's ring
    wrapping several times."""
    tiles = _ring_wrapping_tiles()
    per = -(-tiles * 8192 // len(FORMATS))
    rng = np.random.default_rng(12)
    specs = []
    for i, fmt in enumerate(FORMATS):
        B, _ = synth.GEOMETRY[fmt]
        k = int(rng.integers(8, 40)) * max(B, 64)
        rows = max(1, per // k)
        if fmt == "nvfp4":
            rows = rows // 6 * 6 or 6
        specs.append((fmt, (rows, k), outs[i % len(outs)],
                      synth.payload(fmt, (rows, k), seed=400 + i, ndiv=3 if fmt == "nvfp4" else 1)))
    _batch_and_check(orc, specs, "all formats")
