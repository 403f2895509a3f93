"""Pins for the oracle's IQ2 / IQ3 / IQ1 decoders (iq2_xxs, iq2_xs, iq2_s,
iq3_xxs, iq3_s, iq1_s, iq1_m) and their codebooks, CPU only.

* The codebook fixture (ONNX "DequantizePacked decoding specification",
  "IQ codebooks") against the section's own statements: the row count it
  gives for each table, entries that only select existing values, and
  distinct rows.  The oracle's C expansion is compared with a separate
  Python expansion and with rows decoded by hand from the printed hex.
* An exact-rational restatement of every rule of "IQ2, IQ3, and IQ1
  formats" (every product there is exact in binary32, so each output is the
  exact value rounded once), using its own codebook expansion.
* The sign rules: SP's eighth sign is the parity of the other seven, so a
  lane always has an even number of negative outputs; S uses all eight bits.
* Hand-built blocks with known outputs: IQ1_M's block scale assembled from
  four nibbles, IQ1_S/IQ1_M's +-1/8 shift, IQ3_S's odd multipliers, the
  IQ2_XXS / IQ3_XXS 4-bit scale in the top bits of the sign word.
"""
import struct
from fractions import Fraction

import numpy as np
import pytest

import synth
from test_oracle_formats import ONE_F16, f16, round_f32

IQ = ["gguf:iq2_xxs", "gguf:iq2_xs", "gguf:iq2_s", "gguf:iq3_xxs", "gguf:iq3_s", "gguf:iq1_s", "gguf:iq1_m"]
STATED_ROWS = {"iq2xxs_grid": 256, "iq2xs_grid": 512, "iq2s_grid": 1024, "iq3xxs_grid": 256, "iq3s_grid": 512,
               "iq1s_grid": 2048}


def py_codebooks(orc):
    """Independent expansion: the whole byte string as one little-endian
    integer, entry k = bits [bits*k, bits*k + bits)."""
    out = {}
    for name, (width, bits, _rows, values, packed) in orc.read_codebooks().items():
        big = int.from_bytes(packed.tobytes(), "little")
        n = packed.size * 8 // bits
        ent = [values[(big >> (bits * k)) & ((1 << bits) - 1)] for k in range(n)]
        out[name] = [ent[width * r:width * (r + 1)] for r in range(n // width)]
    return out


def test_codebooks_match_the_stated_row_counts(orc):
    books = orc.read_codebooks()
    assert set(books) == set(STATED_ROWS)
    for name, (width, bits, rows, values, packed) in books.items():
        assert rows == STATED_ROWS[name], name
        assert packed.size * 8 == rows * width * bits, name  # no byte missing or extra
        assert orc.codebook_rows(name) == rows, name
        # every field selects one of the listed values
        big = int.from_bytes(packed.tobytes(), "little")
        assert max((big >> (bits * k)) & ((1 << bits) - 1) for k in range(rows * width)) < len(values), name


def test_codebook_rows_are_distinct(orc):
    for name, rows in py_codebooks(orc).items():
        assert len(set(map(tuple, rows))) == len(rows), name


def test_codebook_expansion_c_vs_python(orc):
    for name, rows in py_codebooks(orc).items():
        for r in range(len(rows)):
            assert orc.codebook_row(name, r) == rows[r], (name, r)


def test_codebook_rows_decoded_by_hand(orc):
    # iq2xxs_grid starts "0000" "0200" "0500": row 1 is byte 0x02 (field 0 =
    # 2 -> 43, fields 1..3 = 0 -> 8) then byte 0x00; row 2 is byte 0x05
    # (fields 1, 1 -> 25, 25).
    assert orc.codebook_row("iq2xxs_grid", 0) == [8] * 8
    assert orc.codebook_row("iq2xxs_grid", 1) == [43] + [8] * 7
    assert orc.codebook_row("iq2xxs_grid", 2) == [25, 25] + [8] * 6
    # iq3xxs_grid: 4-bit fields, 4 per row.  Its first bytes are the first
    # four hex pairs of its first line.
    _, _, _, vals, packed = orc.read_codebooks()["iq3xxs_grid"]
    b0, b1 = int(packed[0]), int(packed[1])
    assert orc.codebook_row("iq3xxs_grid", 0) == [vals[b0 & 15], vals[b0 >> 4], vals[b1 & 15], vals[b1 >> 4]]
    assert set(v for r in range(2048) for v in orc.codebook_row("iq1s_grid", r)) == {-1, 0, 1}


# ---- exact-rational restatement ------------------------------------------
def Hq(b, off):
    return Fraction(struct.unpack_from("<e", bytes(b), off)[0])


def U(b, off, n):
    return sum(b[off + j] << (8 * j) for j in range(n))


def bit(v, j):
    return (v >> j) & 1


def fld(v, k, w):
    return (v >> k) & ((1 << w) - 1)


def signs_S(v):
    return [1 - 2 * bit(v, j) for j in range(8)]


def signs_SP(v):
    low = [bit(v, j) for j in range(7)]
    return [1 - 2 * x for x in low] + [1 - 2 * (sum(low) % 2)]


def exact_iq(fmt, b, G):
    """Exact value of every output of one block, from the rules."""
    b = [int(v) for v in b]
    y = [None] * 256
    if fmt == "gguf:iq1_m":
        w = [U(b, 48 + 2 * k, 2) for k in range(4)]
        hbits = sum((w[k] >> 12) << (4 * k) for k in range(4))
        d = Fraction(struct.unpack("<e", struct.pack("<H", hbits))[0])
    else:
        d = Hq(b, 0)
    for g in range(8):
        for l in range(4):
            i = 4 * g + l
            shifted = False
            if fmt == "gguf:iq2_xxs":
                a = U(b, 6 + 8 * g, 4)
                v, s = G["iq2xxs_grid"][b[2 + 8 * g + l]], signs_SP(fld(a, 7 * l, 7))
                c = d * (Fraction(1, 2) + (a >> 28)) / 4
            elif fmt == "gguf:iq2_xs":
                a = U(b, 2 + 2 * i, 2)
                t = fld(b[66 + g], 4 * (l // 2), 4)
                v, s = G["iq2xs_grid"][a % 512], signs_SP(a // 512)
                c = d * (Fraction(1, 2) + t) / 4
            elif fmt == "gguf:iq2_s":
                r = b[2 + i] + 256 * fld(b[66 + g], 2 * l, 2)
                t = fld(b[74 + g], 4 * (l // 2), 4)
                v, s = G["iq2s_grid"][r], signs_S(b[34 + i])
                c = d * (Fraction(1, 2) + t) / 4
            elif fmt == "gguf:iq3_xxs":
                a = U(b, 66 + 4 * g, 4)
                v = G["iq3xxs_grid"][b[2 + 2 * i]] + G["iq3xxs_grid"][b[3 + 2 * i]]
                s = signs_SP(fld(a, 7 * l, 7))
                c = d * (Fraction(1, 2) + (a >> 28)) / 2
            elif fmt == "gguf:iq3_s":
                r = [b[2 + 2 * i + t] + 256 * bit(b[66 + g], 2 * l + t) for t in (0, 1)]
                v = G["iq3s_grid"][r[0]] + G["iq3s_grid"][r[1]]
                s = signs_S(b[74 + i])
                c = d * (1 + 2 * fld(b[106 + g // 2], 4 * (g % 2), 4))
            elif fmt == "gguf:iq1_s":
                a = U(b, 34 + 2 * g, 2)
                r = b[2 + i] + 256 * fld(a, 3 * l, 3)
                c = d * (2 * fld(a, 12, 3) + 1)
                delta = Fraction(-1, 8) if bit(a, 15) else Fraction(1, 8)
                v, shifted = G["iq1s_grid"][r], True
            else:  # gguf:iq1_m
                a = fld(b[32 + i // 2], 4 * (i % 2), 4)
                r = b[i] + 256 * (a % 8)
                t = fld(w[g // 2], 6 * (g % 2) + 3 * (l // 2), 3)
                c = d * (2 * t + 1)
                delta = Fraction(-1, 8) if bit(a, 3) else Fraction(1, 8)
                v, shifted = G["iq1s_grid"][r], True
            for j in range(8):
                y[8 * i + j] = c * (v[j] + delta) if shifted else c * v[j] * s[j]
    return y


@pytest.mark.parametrize("fmt", IQ)
@pytest.mark.parametrize("dist", ["workload", "bytes"])
def test_exact_rational_restatement(orc, fmt, dist):
    G = py_codebooks(orc)
    B, S = synth.GEOMETRY[fmt]
    nb = 12
    x = synth.payload(fmt, (nb, B), seed=31 + IQ.index(fmt), dist=dist).reshape(nb, S).copy()
    # keep the block scale finite (non-finite scales are covered on the GPU side)
    # (binary16 exponent bits 14..10 all set: clear bit 14)
    if fmt == "gguf:iq1_m":  # bits 15..12 of the scale are the top nibble of byte 55
        x[:, 55] = np.where((x[:, 55] & 0x70) == 0x70, x[:, 55] & 0xBF, x[:, 55])
    else:
        x[:, 1] = np.where((x[:, 1] & 0x7C) == 0x7C, x[:, 1] & 0xBF, x[:, 1])
    for k in range(nb):
        got = orc.decode_block_f32(fmt, x[k].tobytes())
        want = np.array([round_f32(q) for q in exact_iq(fmt, x[k], G)], np.float32)
        # signed zeros: c * v * s with c = +-0 keeps the sign of the product
        assert np.array_equal(got.view(np.uint32) & 0x7FFFFFFF, want.view(np.uint32) & 0x7FFFFFFF), (fmt, k)
        nz = want != 0
        assert np.array_equal(np.signbit(got[nz]), np.signbit(want[nz])), (fmt, k)


# ---- sign rules ------------------------------------------------------------
def test_sp_lanes_have_an_even_number_of_negative_signs(orc):
    # IQ2_XXS with d = 1: lane 0 of group 0 takes its signs from bits 0..6 of
    # the group's 32-bit word; all codebook values are positive.
    for sv in range(128):
        blk = bytearray(66)
        blk[0:2] = ONE_F16
        blk[6:10] = struct.pack("<I", sv)
        y = orc.decode_block_f32("gguf:iq2_xxs", bytes(blk))
        neg = [bool(np.signbit(v)) for v in y[:8]]
        assert neg[:7] == [bool(bit(sv, j)) for j in range(7)], sv
        assert sum(neg) % 2 == 0, sv
        # c = (1 * (0.5 + 0)) * 0.25 and row 0 is all 8s
        assert np.all(np.abs(y[:8]) == 1.0), sv


def test_s_signs_use_all_eight_bits(orc):
    # IQ2_S and IQ3_S take eight independent sign bits: 0xFF negates all 8.
    for fmt, sign_off in (("gguf:iq2_s", 34), ("gguf:iq3_s", 74)):
        blk = bytearray(synth.GEOMETRY[fmt][1])
        blk[0:2] = ONE_F16
        blk[sign_off] = 0xFF
        blk[sign_off + 1] = 0x01
        y = orc.decode_block_f32(fmt, bytes(blk))
        assert np.all(y[:8] < 0) and y[8] < 0 and np.all(y[9:16] > 0), fmt


# ---- hand-built blocks -----------------------------------------------------
def test_iq1_m_block_scale_from_four_nibbles(orc):
    for h in (0x3C00, 0x4500, 0xB800, 0x0001):
        blk = bytearray(56)
        for k in range(4):
            blk[49 + 2 * k] = ((h >> (4 * k)) & 15) << 4
        y = orc.decode_block_f32("gguf:iq1_m", bytes(blk))
        d = float(np.frombuffer(struct.pack("<H", h), np.float16)[0])
        row0 = orc.codebook_row("iq1s_grid", 0)
        # r = 0, t = 0 (c = d), delta = +1/8 everywhere
        want = np.array([np.float32(d) * np.float32(v + 0.125) for v in row0] * 32, np.float32)
        assert np.array_equal(y, want), hex(h)


def test_iq1_m_local_scales_and_shift_sign(orc):
    blk = bytearray(56)
    h = 0x3C00
    w = [((h >> (4 * k)) & 15) << 12 for k in range(4)]
    w[1] |= (5 << 0) | (2 << 3) | (7 << 6) | (1 << 9)  # groups 2 and 3: t = 5, 2, 7, 1
    for k in range(4):
        blk[48 + 2 * k:50 + 2 * k] = struct.pack("<H", w[k])
    blk[32 + 9] = 0x08 | 0x30  # lane i = 18: bit 3 set (delta -1/8); lane 19: r += 256*3
    y = orc.decode_block_f32("gguf:iq1_m", bytes(blk))
    rows = {r: orc.codebook_row("iq1s_grid", r) for r in (0, 768)}
    # group 2: lanes 8, 9 use t = 5 (c = 11), lanes 10, 11 t = 2 (c = 5)
    assert list(y[64:72]) == [11 * (v + 0.125) for v in rows[0]]
    assert list(y[80:88]) == [5 * (v + 0.125) for v in rows[0]]
    # group 4 (lanes 16..19): word 2, t = 0 -> c = 1; lane 18 shifts by -1/8;
    # lane 19 reads row 3*256
    assert list(y[144:152]) == [1 * (v - 0.125) for v in rows[0]]
    assert list(y[152:160]) == [1 * (v + 0.125) for v in rows[768]]
    # group 3: t = 7 for lanes 12, 13 (c = 15), t = 1 for lanes 14, 15 (c = 3)
    assert list(y[96:104]) == [15 * (v + 0.125) for v in rows[0]]
    assert list(y[112:120]) == [3 * (v + 0.125) for v in rows[0]]


def test_iq1_s_scale_index_and_shift(orc):
    blk = bytearray(50)
    blk[0:2] = f16(2.0)
    a = (3 << 12) | (1 << 15) | (5 << 3)  # c = 2 * 7, delta -1/8, lane 1 r += 5*256
    blk[34:36] = struct.pack("<H", a)
    blk[2 + 1] = 7
    y = orc.decode_block_f32("gguf:iq1_s", bytes(blk))
    r0, r1 = orc.codebook_row("iq1s_grid", 0), orc.codebook_row("iq1s_grid", 5 * 256 + 7)
    assert list(y[0:8]) == [14 * (v - 0.125) for v in r0]
    assert list(y[8:16]) == [14 * (v - 0.125) for v in r1]
    assert list(y[32:40]) == [2 * (v + 0.125) for v in r0]  # group 1: a = 0


def test_iq3_s_odd_multipliers(orc):
    blk = bytearray(110)
    blk[0:2] = ONE_F16
    blk[106] = 0xF0  # group 0: field 0 -> c = 1; group 1: field 15 -> c = 31
    blk[66 + 1] = 0b0110  # group 1, lane 0: r[1] += 256; lane 1: r[0] += 256
    y = orc.decode_block_f32("gguf:iq3_s", bytes(blk))
    G = lambda r: orc.codebook_row("iq3s_grid", r)  # noqa: E731
    assert list(y[0:8]) == G(0) + G(0)
    assert list(y[32:40]) == [31 * v for v in G(0) + G(256)]
    assert list(y[40:48]) == [31 * v for v in G(256) + G(0)]


@pytest.mark.parametrize("fmt,cscale", [("gguf:iq2_xxs", 0.25), ("gguf:iq3_xxs", 0.5)])
def test_scale_nibble_in_the_top_bits_of_the_sign_word(orc, fmt, cscale):
    off = 6 if fmt == "gguf:iq2_xxs" else 66
    stride = 8 if fmt == "gguf:iq2_xxs" else 4
    for t in (0, 1, 9, 15):
        blk = bytearray(synth.GEOMETRY[fmt][1])
        blk[0:2] = ONE_F16
        blk[off + stride * 3:off + stride * 3 + 4] = struct.pack("<I", t << 28)
        y = orc.decode_block_f32(fmt, bytes(blk))
        row = orc.codebook_row("iq2xxs_grid", 0) if fmt == "gguf:iq2_xxs" else orc.codebook_row("iq3xxs_grid", 0) * 2
        assert list(y[96:104]) == [(0.5 + t) * cscale * v for v in row], t
        assert list(y[0:8]) == [0.5 * cscale * v for v in row]
