"""Pins for the oracle's other NInfer formats (CPU only): the grouped
signed-integer schemes q2_g64_fp16, q5_g64_fp16, q6_g64_fp16, t2_g128_fp16
and the row-scaled fp8_e4m3fn_row_bf16 / fp8_e4m3fn_row_fp16.

* Geometry against the NInfer "tensor-formats" tables: group size, code
  width and bits/weight (8*S/B = b + 16/G).
* Every code word times special scales against numpy binary32 products,
  with codes packed by an independent Python bit packer; a hand-packed
  5-bit example fixes the bit order.
* Relations the page states: q2_g64_fp16 keeps the Q2_0 grid (q = u - 1) and
  imports gguf Q2_0 blocks without changing code or scale bits, so it
  decodes like gguf:q2_0 on the same bytes; t2's two's-complement words.
* grouped_absmax (NInfer section 7.2) round trips for q5 / q6.
* FP8 rows: all 256 E4M3FN words times BF16 / binary16 multipliers against
  torch's float8_e4m3fn and numpy binary32 products; the row of every code
  and the payload length rule.
"""
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth
from conftest import read_golden
from test_oracle_formats import f16

GROUPED = {"q2_g64_fp16": (2, 64), "q5_g64_fp16": (5, 64), "q6_g64_fp16": (6, 64), "t2_g128_fp16": (2, 128)}
FP8 = ["fp8_e4m3fn_row_bf16", "fp8_e4m3fn_row_fp16"]
SPECIAL_F16 = [0x3C00, 0xC000, 0x0001, 0x8001, 0x0000, 0x8000, 0x7BFF, 0x3555]


def pack_lsb_first(words, width):
    """Independent packer: word k at bits [width*k, width*k + width) of one
    little-endian integer."""
    big = 0
    for k, w in enumerate(words):
        big |= (w & ((1 << width) - 1)) << (width * k)
    n = len(words) * width // 8
    return big.to_bytes(n, "little")


def signed_of(u, width, fmt):
    if fmt == "q2_g64_fp16":
        return u - 1
    return u - (1 << width) if u >= 1 << (width - 1) else u


def test_grouped_geometry_matches_ninfer_table(orc):
    rows = {r[0]: r for r in read_golden("ninfer_grouped_table.txt")}
    for fmt, (width, G) in GROUPED.items():
        _, b, g, qlo, qhi, bpw = rows[fmt]
        B, S, dec = orc.format_info(fmt)
        assert dec and (B, int(b), int(g)) == (G, width, G)
        assert Fraction(8 * S, B) == Fraction(bpw) == Fraction(width) + Fraction(16, G)


@pytest.mark.parametrize("fmt", list(GROUPED))
def test_grouped_every_word_times_special_scales(orc, fmt):
    width, G = GROUPED[fmt]
    words = [k % (1 << width) for k in range(G)]
    codes = pack_lsb_first(words, width)
    for h in SPECIAL_F16:
        scale = np.frombuffer(struct.pack("<H", h), np.float16)[0].astype(np.float32)
        y = orc.decode_block_f32(fmt, struct.pack("<H", h) + codes)
        want = np.array([scale * np.float32(signed_of(u, width, fmt)) for u in words], np.float32)
        assert np.array_equal(y.view(np.uint32), want.view(np.uint32)), (fmt, hex(h))


def test_q5_bit_order_by_hand(orc):
    # codes 1, -1, 0, ...: word 0 = 0b00001 in bits 0..4, word 1 = 0b11111
    # in bits 5..9 -> byte 0 = 0x01 | 0xE0, byte 1 = 0x03
    codes = bytes([0xE1, 0x03]) + bytes(38)
    y = orc.decode_block_f32("q5_g64_fp16", f16(1.0) + codes)
    assert list(y[:3]) == [1.0, -1.0, 0.0] and not y[3:].any()
    # q6: word 0 = -32 (0b100000): bits 0..5 -> byte 0 = 0x20
    y = orc.decode_block_f32("q6_g64_fp16", f16(0.5) + bytes([0x20]) + bytes(47))
    assert y[0] == -16.0 and not y[1:].any()


def test_q2_g64_is_gguf_q2_0_on_identical_bytes(orc):
    x = synth.payload("q2_g64_fp16", (7, 64 * 5), seed=9, dist="bytes")
    for out in ("float32", "bfloat16"):
        a = orc.decode("q2_g64_fp16", (7, 320), x, out)
        b = orc.decode("gguf:q2_0", (7, 320), x, out)
        nan = np.isnan(a.astype(np.float32)) if out == "float32" else np.zeros(a.shape, bool)
        assert np.array_equal(a[~nan], b[~nan])


def test_t2_words(orc):
    # 2-bit two's complement: 0, 1, -2 (0b10, outside the valid language but
    # decoded totally), -1
    y = orc.decode_block_f32("t2_g128_fp16", f16(0.5) + pack_lsb_first([0, 1, 2, 3] * 32, 2))
    assert list(y[:4]) == [0.0, 0.5, -1.0, -0.5]
    assert np.array_equal(y, np.tile(y[:4], 32))


@pytest.mark.parametrize("fmt,G", [("q5_g64_fp16", 64), ("q6_g64_fp16", 64)])
def test_grouped_round_trip(orc, fmt, G):
    rng = np.random.default_rng(22)
    x = (rng.standard_normal((16, 4 * G)) * 0.02).astype(np.float32)
    x[5, G:2 * G] = 0.0
    pay = orc.encode_grouped(fmt, x)
    w = orc.decode(fmt, x.shape, pay, "float32")
    assert orc.encode_grouped(fmt, w).tobytes() == pay.tobytes()
    S = orc.format_info(fmt)[1]
    scales = orc.h2f(pay.reshape(-1, S)[:, 0:2].copy().view("<u2").reshape(-1))
    err = np.abs(x.reshape(-1, G) - w.reshape(-1, G))
    assert (err <= np.abs(scales)[:, None] / 2 * (1 + 1e-6)).all()
    # all-zero group: scale +0, codes 0
    blk = pay.reshape(-1, S)[5 * 4 + 1]
    assert not blk.any()


# ---- row-scaled FP8 ---------------------------------------------------------
def _e4m3fn_all():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()


def _scale_value(fmt, word):
    if fmt == "fp8_e4m3fn_row_bf16":
        return torch.tensor([word], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float().numpy()[0]
    return np.frombuffer(struct.pack("<H", word), np.float16)[0].astype(np.float32)


@pytest.mark.parametrize("fmt", FP8)
def test_fp8_row_all_codes_times_multipliers(orc, fmt):
    c32 = _e4m3fn_all()
    words = ([0x3F80, 0x4000, 0x0001, 0x0080, 0x7F7F, 0x3C23, 0x0000, 0xBF80, 0x7F80]
             if fmt == "fp8_e4m3fn_row_bf16" else [0x3C00, 0x0001, 0x0400, 0x7BFF, 0x2E66, 0x0000, 0xBC00, 0x7C00])
    for w in words:
        s32 = np.float32(_scale_value(fmt, w))
        y = np.array([orc.decode_block_f32(fmt, bytes([c]), float(s32))[0] for c in range(256)], np.float32)
        with np.errstate(over="ignore", invalid="ignore", under="ignore"):
            want = c32 * s32
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(y), nan), (fmt, hex(w))
        assert np.array_equal(y[~nan].view(np.uint32), want[~nan].view(np.uint32)), (fmt, hex(w))


@pytest.mark.parametrize("fmt", FP8)
def test_fp8_row_multiplier_of_each_row(orc, fmt):
    N, K = 3, 5
    codes = np.array([0x38, 0x40, 0xB8, 0x01, 0x7E] * N, np.uint8)  # 1, 2, -1, 2^-9, 448
    words = [0x3F80, 0x4000, 0x3E80] if fmt == "fp8_e4m3fn_row_bf16" else [0x3C00, 0x4000, 0x3400]
    x = np.concatenate([codes, np.array(words, "<u2").view(np.uint8)])
    y = orc.decode(fmt, (N, K), x, "float32")
    base = np.array([1.0, 2.0, -1.0, 2.0 ** -9, 448.0], np.float32)
    for r, m in enumerate((1.0, 2.0, 0.25)):
        assert np.array_equal(y[r], base * np.float32(m)), r
    # rank 1 is one row; rank 3 flattens the leading dimensions into rows
    x1 = np.concatenate([codes[:K], np.array(words[:1], "<u2").view(np.uint8)])
    assert np.array_equal(orc.decode(fmt, (K,), x1, "float32"), base)
    y3 = orc.decode(fmt, (1, N, K), x, "float32")
    assert np.array_equal(y3.reshape(N, K), y)


@pytest.mark.parametrize("fmt", FP8)
def test_fp8_row_length_rule(orc, fmt):
    assert orc.geometry(fmt, (3, 5), 15 + 6) == (15, 3, 3)
    for bad in (15, 15 + 5, 15 + 7, 15 + 8):
        with pytest.raises(orc.OracleError):
            orc.geometry(fmt, (3, 5), bad)
    assert orc.geometry(fmt, (0, 5), 0)[0] == 0
    assert orc.geometry(fmt, (4, 0), 0)[0] == 0
