"""Pins for the oracle's scalar building blocks (CPU only).

binary16 expansion, E8M0 / unsigned-E4M3 half scales, E4M3FN, E2M1 and the
two RNE output casts are checked exhaustively or on large random samples
against library routines (numpy, torch CPU) and the pages' printed values.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden


def _bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def _same_f32(a, b):
    a, b = np.asarray(a, np.float32), np.asarray(b, np.float32)
    nan = np.isnan(a)
    return bool(np.array_equal(nan, np.isnan(b)) and np.array_equal(_bits(a)[~nan], _bits(b)[~nan]))


def test_h2f_exhaustive_vs_numpy(orc):
    words = np.arange(65536, dtype=np.uint16)
    ours = orc.h2f(words)
    ref = words.view(np.float16).astype(np.float32)
    assert _same_f32(ours, ref)
    # signed zeros, the minimum positive subnormal 0x0001 = 2^-24, infinities
    assert _bits(orc.h2f([0x8000]))[0] == 0x80000000
    assert orc.h2f([0x0001])[0] == 2.0 ** -24
    assert np.isinf(orc.h2f([0x7C00, 0xFC00])).all()


def test_e8m0_half_scale_exhaustive(orc):
    # closed form: half scale * V[c] = V[c] * 2^(e-128), rounded once to binary32
    V = [int(r[2]) for r in read_golden("fp4_tables.txt")]
    for e in range(256):
        blk = bytes([e]) + bytes([(c | (c << 4)) for c in range(16)])
        y = orc.decode_block_f32("gguf:mxfp4", blk)
        for c in range(16):
            with np.errstate(over="ignore"):
                want = np.float32(math.ldexp(V[c], e - 128))
            assert _same_f32(y[c], want), (e, c)
            assert _same_f32(y[16 + c], want), (e, c)


def test_e8m0_byte_127_is_unit_scale(orc):
    # gld-kiln worked example: e8m0 byte 127 scales the MXFP4 block by 1.0, so
    # the decoded values are the plain E2M1 values (0, 0.5, ..., 6 and negatives).
    rows = read_golden("kiln_examples.txt")
    e = int([r for r in rows if r[0] == "e8m0"][0][1])
    e2m1 = {int(c): float(v) for c, v in read_golden("e2m1_values.txt")}
    blk = bytes([e]) + bytes([(c | (c << 4)) for c in range(16)])
    y = orc.decode_block_f32("gguf:mxfp4", blk)
    for c in range(16):
        mag = e2m1[c & 7]
        assert y[c] == (-mag if c & 8 else mag)


def test_special_scale_bytes(orc):
    for fmt, byte, val in read_golden("special_scales.txt"):
        e = int(byte, 16)
        if fmt == "gguf:nvfp4":
            assert orc.ue4m3_half(e) == float(val)
            if e in (0x00, 0x7F):
                blk = bytes([e] * 4) + bytes([0x77] * 32)  # code 7 everywhere: V=12
                assert (orc.decode_block_f32("gguf:nvfp4", blk) == 0).all()
        else:
            got = np.float32(orc.e8m0_half(e))
            want = np.uint32(int(val, 16)).view(np.float32) if val.startswith("0x") else np.float32(val)
            assert _bits(got) == _bits(want)


def test_ue4m3_half_scale_exhaustive(orc):
    # closed form from the NVFP4 rule, evaluated in exact rationals
    for e in range(256):
        E, m = (e >> 3) & 15, e % 8
        if e in (0, 127):
            want = Fraction(0)
        elif E == 0:
            want = Fraction(m, 1024)
        else:
            want = (1 + Fraction(m, 8)) * Fraction(2) ** (E - 8)
        assert Fraction(orc.ue4m3_half(e)) == want, e


def test_e4m3fn_all_words_vs_torch(orc):
    words = torch.arange(256, dtype=torch.uint8)
    ref = words.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    ours = np.array([orc.e4m3fn(w) for w in range(256)], np.float32)
    assert _same_f32(ours, ref)
    assert np.isnan(ours[[0x7F, 0xFF]]).all()
    assert _bits(ours[0x80]) == 0x80000000  # signed zero


def test_ue4m3_half_is_half_of_e4m3fn_on_valid_words(orc):
    # For bytes 0x01..0x7e the unsigned-E4M3 half scale is E4M3FN / 2.
    for e in range(1, 0x7F):
        assert orc.ue4m3_half(e) == orc.e4m3fn(e) / 2, e


def test_e2m1_words(orc):
    table = {int(c): float(v) for c, v in read_golden("e2m1_values.txt")}
    for c in range(16):
        v = orc.e2m1(c)
        mag = table[c & 7]
        if c & 8:
            assert v == -mag and math.copysign(1.0, v) == -1.0
        else:
            assert v == mag and math.copysign(1.0, v) == 1.0
    # The doubled table V of the GGUF block-floating formats is 2 * E2M1 with
    # both zeros positive.
    for idx, _iq4, V in read_golden("fp4_tables.txt"):
        i = int(idx)
        assert int(V) == (0 if i == 8 else int(2 * orc.e2m1(i)))


def _special_f32_patterns():
    pats = [0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0x7F800001, 0xFFC00001,
            0x7F7FFFFF, 0xFF7FFFFF, 0x00000001, 0x80000001, 0x007FFFFF, 0x00800000]
    # bf16 ties / near-ties and binary16 boundaries: max, overflow midpoint,
    # smallest normal/subnormal and their half-way points
    for base in (0x3F800000, 0x3F810000, 0x40490FDB, 0x477FE000, 0x477FF000, 0x477FEFFF,
                 0x38800000, 0x33800000, 0x33000000, 0x33000001, 0x32FFFFFF, 0x387FC000,
                 0x387FE000, 0x33C00000):
        for d in (-1, 0, 1, 0x7FFF, 0x8000, 0x8001, 0x0FFF, 0x1000, 0x1001):
            for s in (0, 0x80000000):
                pats.append(((base + d) & 0x7FFFFFFF) | s)
    return np.array(pats, dtype=np.uint32)


def test_bf16_cast_vs_torch(orc):
    rng = np.random.default_rng(11)
    pats = np.concatenate([_special_f32_patterns(), rng.integers(0, 2**32, size=1 << 22, dtype=np.uint32)])
    ours = orc.f32_to_bf16(pats)
    ref = torch.from_numpy(pats.view(np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()
    nan = np.isnan(pats.view(np.float32))
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN
    assert ((ours[nan] & 0x7F80) == 0x7F80).all() and ((ours[nan] & 0x7F) != 0).all()


def test_f16_cast_vs_numpy_and_torch(orc):
    rng = np.random.default_rng(12)
    pats = np.concatenate([_special_f32_patterns(), rng.integers(0, 2**32, size=1 << 22, dtype=np.uint32)])
    # also dense coverage of the binary16 range and the subnormal range
    pats = np.concatenate([pats, rng.integers(0x33000000, 0x47800000, size=1 << 20, dtype=np.uint32)])
    ours = orc.f32_to_f16(pats)
    with np.errstate(over="ignore"):
        ref_np = pats.view(np.float32).astype(np.float16).view(np.uint16)
    ref_t = torch.from_numpy(pats.view(np.float32)).to(torch.float16).view(torch.uint16).numpy()
    nan = np.isnan(pats.view(np.float32))
    assert np.array_equal(ours[~nan], ref_np[~nan])
    assert np.array_equal(ours[~nan], ref_t[~nan])
    assert ((ours[nan] & 0x7C00) == 0x7C00).all() and ((ours[nan] & 0x3FF) != 0).all()
