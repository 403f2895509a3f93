"""Pins for the oracle's decoders of the remaining simple gguf profiles
(q4_1, q5_0, q5_1, q8_1, q8_k, q2_k, q3_k, q5_k, iq4_xs, tq1_0, tq2_0,
q1_0, q2_0), CPU only.

* an exact-rational restatement of each rule of the ONNX "DequantizePacked
  decoding specification", "Mathematical decoding rules" (every inner
  product of these formats is exact in binary32, so each output is the
  exact value rounded once);
* hand-built blocks with known integer outputs (the K-quant scale layouts,
  the 1- and 2-bit plane orders, the IQ4_XS sub-scales);
* relations the rules imply: cached sum fields are ignored (Q8_1, Q8_K),
  Q8_1 is Q8_0 with an extra field, Q4_1 with m = -8d is Q4_0, Q5_0 with no
  high bits is Q4_0 shifted by 8d;
* TQ1_0's wrapped-byte rule is the base-3 expansion of b/256: for every
  byte, the p-th output is the p-th base-3 digit of b/256 minus one.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest

import synth
from test_oracle_formats import IQ4, ONE_F16, f16, planes, round_f32, s8

NEXT = ["gguf:q4_1", "gguf:q5_0", "gguf:q5_1", "gguf:q8_1", "gguf:q8_k", "gguf:q2_k", "gguf:q3_k",
        "gguf:q5_k", "gguf:iq4_xs", "gguf:tq1_0", "gguf:tq2_0", "gguf:q1_0", "gguf:q2_0"]


def Hq(b, off):
    return Fraction(struct.unpack_from("<e", bytes(b), off)[0])


def Fq(b, off):
    return Fraction(struct.unpack_from("<f", bytes(b), off)[0])


def U(b, off, n):
    return sum(b[off + j] << (8 * j) for j in range(n))


def kq_am(s, k):
    if k < 4:
        return s[k] & 63, s[k + 4] & 63
    return (s[k + 4] & 15) + 16 * (s[k - 4] >> 6), (s[k + 4] >> 4) + 16 * (s[k] >> 6)


def exact_next(fmt, b):
    """Exact value of every output of one block, from the rules."""
    b = list(b)
    if fmt in ("gguf:q4_1", "gguf:q5_0", "gguf:q5_1"):
        aff = fmt != "gguf:q5_0"
        o = 4 if aff else 2
        d = Hq(b, 0)
        m = Hq(b, 2) if aff else 0
        if fmt == "gguf:q4_1":
            v = planes(b[4:20], 4, 16)
        else:
            high = U(b, o, 4)
            v = [x + 16 * ((high >> j) & 1) for j, x in enumerate(planes(b[o + 4:o + 20], 4, 16))]
        return [d * x + m for x in v] if aff else [d * (x - 16) for x in v]
    if fmt == "gguf:q8_1":
        return [Hq(b, 0) * s8(b[4 + j]) for j in range(32)]
    if fmt == "gguf:q8_k":
        return [Fq(b, 0) * s8(b[4 + j]) for j in range(256)]
    if fmt == "gguf:q2_k":
        v, d, dm = planes(b[16:80], 2, 32), Hq(b, 80), Hq(b, 82)
        return [d * (b[j // 16] & 15) * v[j] - dm * (b[j // 16] >> 4) for j in range(256)]
    if fmt == "gguf:q3_k":
        v, h = planes(b[32:96], 2, 32), planes(b[0:32], 1, 32)
        l, a = planes(b[96:104], 4, 8), planes(b[104:108], 2, 4)
        d = Hq(b, 108)
        return [d * (l[j // 16] + 16 * a[j // 16] - 32) * (v[j] - 4 * (1 - h[j])) for j in range(256)]
    if fmt == "gguf:q5_k":
        d, dm = Hq(b, 0), Hq(b, 2)
        v, hb = planes(b[48:176], 4, 32), planes(b[16:48], 1, 32)
        out = []
        for j in range(256):
            a, m = kq_am(b[4:16], j // 32)
            out.append(d * a * (v[j] + 16 * hb[j]) - dm * m)
        return out
    if fmt == "gguf:iq4_xs":
        d, high, v = Hq(b, 0), U(b, 2, 2), planes(b[8:136], 4, 16)
        sc = [((b[4 + k // 2] >> (4 * (k % 2))) & 15) + 16 * ((high >> (2 * k)) & 3) - 32 for k in range(8)]
        return [d * sc[j // 32] * IQ4[v[j]] for j in range(256)]
    if fmt == "gguf:tq1_0":
        d, out = Hq(b, 52), []
        for start, width, count in ((0, 32, 5), (32, 16, 5), (48, 4, 4)):
            for p in range(count):
                for j in range(width):
                    out.append(d * ((3 * ((b[start + j] * 3 ** p) % 256)) // 256 - 1))
        return out
    if fmt == "gguf:tq2_0":
        return [Hq(b, 64) * (x - 1) for x in planes(b[0:64], 2, 32)]
    if fmt == "gguf:q1_0":
        d = Hq(b, 0)
        return [d if (b[2 + j // 8] >> (j % 8)) & 1 else -d for j in range(128)]
    if fmt == "gguf:q2_0":
        return [Hq(b, 0) * (x - 1) for x in planes(b[2:18], 2, 1)]
    raise ValueError(fmt)


def _finite(fmt, blk):
    offs = synth.F16_SCALES.get(fmt, ())
    if fmt == "gguf:q8_k":
        return (blk[3] & 0x7F) != 0x7F or (blk[2] & 0x80) == 0
    return all((blk[o + 1] & 0x7C) != 0x7C for o in offs)


@pytest.mark.parametrize("fmt", NEXT)
@pytest.mark.parametrize("dist", ["workload", "bytes"])
def test_exact_rational_restatement(orc, fmt, dist):
    B, S, dec = orc.format_info(fmt)
    assert dec
    x = synth.payload(fmt, (1, B * 24), seed=303, dist=dist)
    checked = 0
    for i in range(24):
        blk = x[i * S:(i + 1) * S].tobytes()
        if not _finite(fmt, blk):
            continue
        y = orc.decode_block_f32(fmt, blk)
        ex = exact_next(fmt, blk)
        for j in range(B):
            want = round_f32(ex[j])
            assert y[j] == want or (np.isinf(y[j]) and np.isinf(want) and np.sign(y[j]) == np.sign(want)), \
                (fmt, i, j, y[j], want)
        checked += 1
    assert checked >= 10


def test_cached_sums_are_ignored(orc):
    rng = np.random.default_rng(8)
    base = bytearray(rng.integers(0, 256, 36, dtype=np.uint8).tobytes())
    base[0:2] = ONE_F16
    y0 = orc.decode_block_f32("gguf:q8_1", bytes(base))
    for s in (b"\x00\x00", b"\xff\xff", b"\x00\x7c", b"\x01\x7e"):  # +0, NaN, inf, NaN
        base[2:4] = s
        assert np.array_equal(orc.decode_block_f32("gguf:q8_1", bytes(base)), y0)
    # Q8_1 is Q8_0 with the extra cached field
    q80 = bytes(base[0:2]) + bytes(base[4:36])
    assert np.array_equal(orc.decode_block_f32("gguf:q8_0", q80), y0)
    kb = bytearray(rng.integers(0, 256, 292, dtype=np.uint8).tobytes())
    kb[0:4] = np.array([0.5], "<f4").tobytes()
    k0 = orc.decode_block_f32("gguf:q8_k", bytes(kb))
    kb[260:292] = bytes(32)
    assert np.array_equal(orc.decode_block_f32("gguf:q8_k", bytes(kb)), k0)
    assert list(k0) == [0.5 * s8(v) for v in kb[4:260]]


def test_q4_1_with_minus_8d_is_q4_0(orc):
    q = bytes([(j | ((15 - j) << 4)) for j in range(16)])
    for d in (1.0, -2.0, 0.125, 3.5):
        a = orc.decode_block_f32("gguf:q4_1", f16(d) + f16(-8 * d) + q)
        b = orc.decode_block_f32("gguf:q4_0", f16(d) + q)
        assert np.array_equal(a, b), d


def test_q5_0_without_high_bits_is_q4_0_shifted(orc):
    q = bytes([(j | ((15 - j) << 4)) for j in range(16)])
    a = orc.decode_block_f32("gguf:q5_0", ONE_F16 + bytes(4) + q)
    b = orc.decode_block_f32("gguf:q4_0", ONE_F16 + q)
    assert list(a) == [v - 8 for v in b]


def test_q5_high_bits_hand_built(orc):
    q = bytes([(j | ((15 - j) << 4)) for j in range(16)])
    high = 0b10110000_00000000_00000001_10000011
    order = [j for j in range(16)] + [15 - j for j in range(16)]  # P(q,4,16)
    hb = np.array([high], "<u4").tobytes()
    y0 = orc.decode_block_f32("gguf:q5_0", ONE_F16 + hb + q)
    y1 = orc.decode_block_f32("gguf:q5_1", f16(2.0) + f16(-1.0) + hb + q)
    for j in range(32):
        v = order[j] + 16 * ((high >> j) & 1)
        assert y0[j] == v - 16 and y1[j] == 2 * v - 1


def test_q2_k_hand_built(orc):
    sc = [(a | (m << 4)) for a, m in zip(range(16), [15 - k for k in range(16)])]
    v = [(j * 3 + j // 7) % 4 for j in range(256)]
    q = [0] * 64
    for j in range(256):  # inverse of P(q,2,32): group j//128, plane (j%128)//32, byte j%32
        q[32 * (j // 128) + j % 32] |= v[j] << (2 * ((j % 128) // 32))
    blk = bytes(sc) + bytes(q) + ONE_F16 + f16(0.5)
    y = orc.decode_block_f32("gguf:q2_k", blk)
    assert list(y) == [(sc[j // 16] & 15) * v[j] - 0.5 * (sc[j // 16] >> 4) for j in range(256)]


def test_q3_k_hand_built(orc):
    s6 = [(k * 11 + 5) % 64 for k in range(16)]  # l + 16a, l 4 bits, a 2 bits
    lb, ab = [0] * 8, [0] * 4
    for k in range(16):  # inverses of P(b[96:104],4,8) and P(b[104:108],2,4)
        lb[k % 8] |= (s6[k] & 15) << (4 * (k // 8))
        ab[k % 4] |= (s6[k] >> 4) << (2 * (k // 4))
    v = [(j * 5 + j // 9) % 4 for j in range(256)]
    h = [(j // 3) % 2 for j in range(256)]
    q, mask = [0] * 64, [0] * 32
    for j in range(256):
        q[32 * (j // 128) + j % 32] |= v[j] << (2 * ((j % 128) // 32))
        mask[j % 32] |= h[j] << (j // 32)  # P(mask,1,32): plane j//32, byte j%32
    blk = bytes(mask) + bytes(q) + bytes(lb) + bytes(ab) + ONE_F16
    y = orc.decode_block_f32("gguf:q3_k", blk)
    assert list(y) == [(s6[j // 16] - 32) * (v[j] - 4 * (1 - h[j])) for j in range(256)]


def test_q5_k_hand_built(orc):
    from test_oracle_formats import _pack_q4_k_scales
    a = [5, 63, 17, 32, 61, 18, 47, 33]
    m = [9, 40, 0, 63, 50, 3, 29, 62]
    v = [(j * 5 + j // 32) % 16 for j in range(256)]
    hb = [(j // 5) % 2 for j in range(256)]
    q, high = [0] * 128, [0] * 32
    for j in range(256):
        q[32 * (j // 64) + j % 32] |= v[j] << (4 * ((j % 64) // 32))
        high[j % 32] |= hb[j] << (j // 32)
    blk = ONE_F16 + ONE_F16 + _pack_q4_k_scales(a, m) + bytes(high) + bytes(q)
    y = orc.decode_block_f32("gguf:q5_k", blk)
    assert list(y) == [a[j // 32] * (v[j] + 16 * hb[j]) - m[j // 32] for j in range(256)]


def test_iq4_xs_hand_built(orc):
    s6 = [0, 63, 31, 32, 1, 62, 17, 45]  # sub-scale + 32 for each of the 8 sub-blocks
    high = sum((s >> 4) << (2 * k) for k, s in enumerate(s6))
    lows = bytes([(s6[2 * i] & 15) | ((s6[2 * i + 1] & 15) << 4) for i in range(4)])
    v = [(j * 7 + j // 11) % 16 for j in range(256)]
    q = [0] * 128
    for j in range(256):  # inverse of P(q,4,16): group j//32, plane (j%32)//16, byte j%16
        q[16 * (j // 32) + j % 16] |= v[j] << (4 * ((j % 32) // 16))
    blk = ONE_F16 + np.array([high], "<u2").tobytes() + lows + bytes(q)
    y = orc.decode_block_f32("gguf:iq4_xs", blk)
    assert list(y) == [(s6[j // 32] - 32) * IQ4[v[j]] for j in range(256)]


def _base3_digits(num, den, n):
    x, out = Fraction(num, den), []
    for _ in range(n):
        x *= 3
        dgt = math.floor(x)
        out.append(dgt)
        x -= dgt
    return out


def test_tq1_0_is_base3_expansion(orc):
    # every byte in every lane position: outputs are base-3 digits of b/256, minus one
    for b0 in range(0, 256, 32):
        bs = [(b0 + i) % 256 for i in range(54)]
        blk = bytes(bs[:52]) + ONE_F16
        y = orc.decode_block_f32("gguf:tq1_0", blk)
        n = 0
        for start, width, count in ((0, 32, 5), (32, 16, 5), (48, 4, 4)):
            for p in range(count):
                for j in range(width):
                    assert y[n] == _base3_digits(bs[start + j], 256, 5)[p] - 1, (b0, start, p, j)
                    n += 1
        assert n == 256


def test_tq2_0_and_q2_0_plane_orders(orc):
    # tq2_0: P(q,2,32); byte j of each 32-byte group holds 4 consecutive planes
    q = bytes([0b11_10_01_00] * 64)  # planes 0..3 = 0,1,2,3
    y = orc.decode_block_f32("gguf:tq2_0", q + ONE_F16)
    assert list(y) == [((j % 128) // 32) - 1 for j in range(256)]
    # q2_0: P(q,2,1): each byte's four 2-bit codes are consecutive outputs
    y = orc.decode_block_f32("gguf:q2_0", ONE_F16 + bytes([0b00_01_10_11] * 16))
    assert list(y) == [2, 1, 0, -1] * 16


def test_q1_0_signs_without_multiplication(orc):
    bits = bytes([0b1010_0101, 0xFF, 0x00, 0x0F] * 4)
    for d in (1.5, -0.25, 0.0, -0.0):
        y = orc.decode_block_f32("gguf:q1_0", f16(d) + bits)
        for j in range(128):
            want = d if (bits[j // 8] >> (j % 8)) & 1 else -d
            assert y[j] == want and math.copysign(1, y[j]) == math.copysign(1, want)
