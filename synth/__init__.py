"""Seeded synthetic payload generators for packed quantized weights.

This module only draws random field values and lays them out as bytes; it
contains none of the decode arithmetic.  It is shared by the tests (which
feed the same bytes to the CPU oracle and the CUDA library) and by the
benchmark.  Every generator is a pure function of (shape, seed).

Field distributions follow the benchmark workloads:
  * gguf:q8_0  -- per block one binary16 scale drawn log-uniform in
    [1e-3, 1e-1], 32 signed bytes uniform in [-127, 127];
  * gguf:q4_0, q4_g64_fp16, gguf:iq4_nl -- binary16 scales |N(0,0.02)|+1e-4,
    code bytes uniform (every nibble value 0..15 equally likely);
  * gguf:q4_k, gguf:q6_k -- binary16 d/dmin |N(0,0.01)|, every other byte
    (packed 6-bit sub-scales and minima, signed 8-bit sub-scales, quant
    nibbles and 2-bit planes) uniform;
  * gguf:mxfp4 -- exponent byte uniform in [118, 130], code bytes uniform;
  * nvfp4 -- E4M3FN scale bytes uniform over 0x00..0x7e (every valid
    nonnegative finite word), code bytes uniform, one FP32 divisor
    d_w = binary32(2688 / binary32(amax)) with amax = 0.1 (448*6/amax);
  * gguf:nvfp4 -- scale bytes uniform over 0x00..0x7e, codes uniform;
  * the other gguf formats (q4_1, q5_0, q5_1, q8_1, q8_k, q2_k, q3_k, q5_k,
    iq4_xs, tq1_0, tq2_0, q1_0, q2_0, iq2_xxs, iq2_xs, iq2_s, iq3_xxs, iq3_s,
    iq1_s, iq1_m, and NInfer's q2/q5/q6_g64_fp16, t2_g128_fp16) -- binary16
    scales |N(0,0.02)|+1e-4 (t2: only the valid words 0, 1, 3; iq1_m: its scale's
    four nibbles in the top bits of the four 16-bit words at byte 48),
    minima |N(0,0.01)|, q8_k's binary32 scale likewise, codes in [-127, 127]
    for q8_k, every other byte uniform;
  * fp8_e4m3fn_row_bf16 / _fp16 -- codes uniform over the 254 non-NaN
    E4M3FN words, then one positive row multiplier |N(0,0.02)|+1e-4 per
    row (BF16 or binary16);
  * "bytes" -- every byte uniform over 0..255 (exercises special scales:
    binary16 infinities/NaNs, E4M3FN NaN words, E8M0 extremes).

Blocks are row-contiguous along the last dimension (row-major shapes).
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np

# (B, S) of the formats generated here.  Geometry only; no decode rules.
GEOMETRY = {
    "gguf:q8_0": (32, 34), "q8_g32_fp16": (32, 34), "gguf:q4_0": (32, 18),
    "gguf:iq4_nl": (32, 18), "q4_g64_fp16": (64, 34), "gguf:q4_k": (256, 144),
    "gguf:q6_k": (256, 210), "gguf:mxfp4": (32, 17), "gguf:nvfp4": (64, 36),
    "nvfp4": (64, 36),
    "gguf:q4_1": (32, 20), "gguf:q5_0": (32, 22), "gguf:q5_1": (32, 24), "gguf:q8_1": (32, 36),
    "gguf:q8_k": (256, 292), "gguf:q2_k": (256, 84), "gguf:q3_k": (256, 110), "gguf:q5_k": (256, 176),
    "gguf:iq4_xs": (256, 136), "gguf:tq1_0": (256, 54), "gguf:tq2_0": (256, 66), "gguf:q1_0": (128, 18),
    "gguf:q2_0": (64, 18),
    "gguf:iq2_xxs": (256, 66), "gguf:iq2_xs": (256, 74), "gguf:iq2_s": (256, 82), "gguf:iq3_xxs": (256, 98),
    "gguf:iq3_s": (256, 110), "gguf:iq1_s": (256, 50), "gguf:iq1_m": (256, 56),
    "q2_g64_fp16": (64, 18), "q5_g64_fp16": (64, 42), "q6_g64_fp16": (64, 50), "t2_g128_fp16": (128, 34),
    "fp8_e4m3fn_row_bf16": (1, 1), "fp8_e4m3fn_row_fp16": (1, 1),
}
# Formats whose payload ends with one 16-bit multiplier per row (after the
# row-major code plane).
ROW_SCALED = ("fp8_e4m3fn_row_bf16", "fp8_e4m3fn_row_fp16")

# Byte offsets of the binary16 scale fields of the other gguf formats; their
# workload recipe draws these from |N(0,0.02)|+1e-4 (minima |N(0,0.01)|) and
# every other byte uniformly.  q8_k's scale is one binary32 at offset 0.
F16_SCALES = {
    "gguf:q4_1": (0, 2), "gguf:q5_0": (0,), "gguf:q5_1": (0, 2), "gguf:q8_1": (0,), "gguf:q2_k": (80, 82),
    "gguf:q3_k": (108,), "gguf:q5_k": (0, 2), "gguf:iq4_xs": (0,), "gguf:tq1_0": (52,), "gguf:tq2_0": (64,),
    "gguf:q1_0": (0,), "gguf:q2_0": (0,),
    "gguf:iq2_xxs": (0,), "gguf:iq2_xs": (0,), "gguf:iq2_s": (0,), "gguf:iq3_xxs": (0,), "gguf:iq3_s": (0,),
    "gguf:iq1_s": (0,),
}

NVFP4_AMAX = 0.1


def _nblocks(fmt: str, shape) -> int:
    B, _ = GEOMETRY[fmt]
    n = 1
    for s in shape[:-1]:
        n *= int(s)
    K = int(shape[-1])
    if K % B:
        raise ValueError(f"{fmt}: last dim {K} not a multiple of {B}")
    return n * (K // B)


def _u8(rng, shape) -> np.ndarray:
    return rng.integers(0, 256, size=shape, dtype=np.uint8)


def _f16_bytes(values: np.ndarray) -> np.ndarray:
    """binary16 (numpy RNE conversion) as little-endian byte pairs, shape [n, 2]."""
    return values.astype(np.float16).astype("<f2").view(np.uint8).reshape(-1, 2)


def nvfp4_divisor(amax: float = NVFP4_AMAX) -> np.float32:
    """The global FP32 divisor of the workload: binary32(448*6 / binary32(amax))."""
    return np.float32(np.float32(2688.0) / np.float32(amax))


def nvfp4_divisors(ndiv: int, seed: int) -> np.ndarray:
    """`ndiv` FP32 divisors: the workload's d_w first, then 2688/U(0.01, 1)."""
    rng = np.random.default_rng(seed + 7919)
    extra = np.float32(2688.0) / rng.uniform(0.01, 1.0, size=max(0, ndiv - 1)).astype(np.float32)
    return np.concatenate([np.array([nvfp4_divisor()], np.float32), extra.astype(np.float32)])


def payload(fmt: str, shape, seed: int, dist: str = "workload", ndiv: int = 1) -> np.ndarray:
    """Packed payload bytes (uint8, flat) for `fmt` with logical `shape`.

    dist="workload" uses the benchmark field distributions above;
    dist="bytes" draws every byte uniformly (including scale fields).
    For nvfp4, `ndiv` FP32 divisors follow the blocks (none when empty).
    """
    rng = np.random.default_rng(seed)
    nb = _nblocks(fmt, shape)
    B, S = GEOMETRY[fmt]
    blk = _u8(rng, (nb, S))
    rows = int(np.prod(shape[:-1], dtype=np.int64))
    if dist == "bytes":
        out = blk.reshape(-1)
        if fmt == "nvfp4" and nb:
            out = np.concatenate([out, nvfp4_divisors(ndiv, seed).astype("<f4").view(np.uint8)])
        if fmt in ROW_SCALED and nb:
            out = np.concatenate([out, _u8(rng, 2 * rows)])
        return out
    if dist != "workload":
        raise ValueError(dist)
    if fmt in ("gguf:q8_0", "q8_g32_fp16"):
        d = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), size=nb))
        blk[:, 0:2] = _f16_bytes(d)
        blk[:, 2:34] = rng.integers(-127, 128, size=(nb, 32), dtype=np.int8).view(np.uint8)
    elif fmt in ("gguf:q4_0", "gguf:iq4_nl", "q4_g64_fp16"):
        d = np.abs(rng.normal(0.0, 0.02, size=nb)) + 1e-4
        blk[:, 0:2] = _f16_bytes(d)
    elif fmt == "gguf:q4_k":
        d = np.abs(rng.normal(0.0, 0.01, size=(nb, 2)))
        blk[:, 0:4] = _f16_bytes(d.reshape(-1)).reshape(nb, 4)
    elif fmt == "gguf:q6_k":
        d = np.abs(rng.normal(0.0, 0.01, size=nb))
        blk[:, 208:210] = _f16_bytes(d)
    elif fmt == "gguf:mxfp4":
        blk[:, 0] = rng.integers(118, 131, size=nb, dtype=np.uint8)
    elif fmt in ("gguf:nvfp4", "nvfp4"):
        blk[:, 0:4] = rng.integers(0, 0x7F, size=(nb, 4), dtype=np.uint8)
    elif fmt in F16_SCALES:
        for i, off in enumerate(F16_SCALES[fmt]):
            sd = 0.02 if i == 0 else 0.01
            blk[:, off:off + 2] = _f16_bytes(np.abs(rng.normal(0.0, sd, size=nb)) + (1e-4 if i == 0 else 0.0))
    elif fmt == "gguf:iq1_m":
        # the binary16 block scale is split over the top 4 bits of the four
        # 16-bit words at byte 48 (nibble k of the scale in word k)
        h = (np.abs(rng.normal(0.0, 0.02, size=nb)) + 1e-4).astype(np.float16).view(np.uint16).astype(np.uint32)
        for k in range(4):
            blk[:, 49 + 2 * k] = (blk[:, 49 + 2 * k] & 0x0F) | (((h >> (4 * k)) & 15) << 4).astype(np.uint8)
    elif fmt in ("q2_g64_fp16", "q5_g64_fp16", "q6_g64_fp16", "t2_g128_fp16"):
        blk[:, 0:2] = _f16_bytes(np.abs(rng.normal(0.0, 0.02, size=nb)) + 1e-4)
        if fmt == "t2_g128_fp16":  # valid ternary words only: 0, 1, 3 (0b10 is outside the format)
            w = rng.choice(np.array([0, 1, 3], np.uint8), size=(nb, 32, 4))
            blk[:, 2:34] = w[..., 0] | (w[..., 1] << 2) | (w[..., 2] << 4) | (w[..., 3] << 6)
    elif fmt in ROW_SCALED:
        # every valid E4M3FN word (0x7f and 0xff are NaN words), positive
        # row multipliers |N(0,0.02)| + 1e-4 as BF16 or binary16
        codes = rng.integers(0, 254, size=nb, dtype=np.uint8)
        blk[:, 0] = np.where(codes >= 0x7F, codes + 1, codes).astype(np.uint8)
        sc = (np.abs(rng.normal(0.0, 0.02, size=rows)) + 1e-4).astype(np.float32)
        if fmt == "fp8_e4m3fn_row_fp16":
            words = sc.astype(np.float16).view(np.uint16)
        else:  # the high half of the binary32 pattern
            words = (sc.view(np.uint32) >> 16).astype(np.uint16)
        return np.concatenate([blk.reshape(-1), words.astype("<u2").view(np.uint8)]) if nb else blk.reshape(-1)
    elif fmt == "gguf:q8_k":
        d = (np.abs(rng.normal(0.0, 0.02, size=nb)) + 1e-4).astype("<f4")
        blk[:, 0:4] = d.view(np.uint8).reshape(nb, 4)
        blk[:, 4:260] = rng.integers(-127, 128, size=(nb, 256), dtype=np.int8).view(np.uint8)
    else:
        raise ValueError(fmt)
    out = blk.reshape(-1)
    if fmt == "nvfp4" and nb:
        out = np.concatenate([out, nvfp4_divisors(ndiv, seed).astype("<f4").view(np.uint8)])
    return out


def sha256(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).view(np.uint8).data).hexdigest()


# --------------------------------------------------------------------------
# Benchmark workloads.
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class TensorSpec:
    name: str
    fmt: str
    shape: tuple
    seed: int
    out_dtype: str


def llama3_8b_tensors() -> list[TensorSpec]:
    """Whole-model decode: Llama-3-8B-shaped weights.

    32 layers of attention q/o [4096,4096] and k/v [1024,4096] in gguf:q4_k,
    FFN gate/up [14336,4096] and down [4096,14336] in gguf:q6_k, and one
    embedding [128256,4096] in gguf:q8_0; 225 tensors, all decoded to bf16.
    Tensor i uses seed 1000 + i.
    """
    specs = []
    i = 0
    for layer in range(32):
        for nm, shp in (("q", (4096, 4096)), ("k", (1024, 4096)), ("v", (1024, 4096)), ("o", (4096, 4096))):
            specs.append(TensorSpec(f"layers.{layer}.attn.{nm}", "gguf:q4_k", shp, 1000 + i, "bfloat16"))
            i += 1
        for nm, shp in (("gate", (14336, 4096)), ("up", (14336, 4096)), ("down", (4096, 14336))):
            specs.append(TensorSpec(f"layers.{layer}.ffn.{nm}", "gguf:q6_k", shp, 1000 + i, "bfloat16"))
            i += 1
    specs.append(TensorSpec("embed", "gguf:q8_0", (128256, 4096), 1000 + i, "bfloat16"))
    return specs


# Single-format workloads: (label, format, shape, seed, output dtype).
WORKLOADS = [
    ("q8_0[256,4096]->f32", "gguf:q8_0", (256, 4096), 0, "float32"),
    ("q4_0[4096,4096]->bf16", "gguf:q4_0", (4096, 4096), 1, "bfloat16"),
    ("q4_g64_fp16[4096,4096]->bf16", "q4_g64_fp16", (4096, 4096), 2, "bfloat16"),
    ("q4_k[14336,4096]->f16", "gguf:q4_k", (14336, 4096), 3, "float16"),
    ("q6_k[14336,4096]->f16", "gguf:q6_k", (14336, 4096), 4, "float16"),
    ("nvfp4[8192,28672]->bf16", "nvfp4", (8192, 28672), 5, "bfloat16"),
    ("mxfp4[8192,28672]->bf16", "gguf:mxfp4", (8192, 28672), 6, "bfloat16"),
    ("iq4_nl[8192,28672]->bf16", "gguf:iq4_nl", (8192, 28672), 7, "bfloat16"),
]

# The other gguf and NInfer formats, each on one Llama-3-8B FFN-shaped tensor
# [14336, 4096] decoded to bf16; seeds 100 + index.
NEXT_FORMATS = ["gguf:q4_1", "gguf:q5_0", "gguf:q5_1", "gguf:q8_1", "gguf:q8_k", "gguf:q2_k", "gguf:q3_k",
                "gguf:q5_k", "gguf:iq4_xs", "gguf:tq1_0", "gguf:tq2_0", "gguf:q1_0", "gguf:q2_0",
                "gguf:iq2_xxs", "gguf:iq2_xs", "gguf:iq2_s", "gguf:iq3_xxs", "gguf:iq3_s", "gguf:iq1_s", "gguf:iq1_m",
                "q2_g64_fp16", "q5_g64_fp16", "q6_g64_fp16", "t2_g128_fp16", "fp8_e4m3fn_row_bf16",
                "fp8_e4m3fn_row_fp16"]
NEXT_WORKLOADS = [(f"{f.split(':')[-1]}[14336,4096]->bf16", f, (14336, 4096), 100 + i, "bfloat16")
                  for i, f in enumerate(NEXT_FORMATS)]
