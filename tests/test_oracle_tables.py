"""Pins for the oracle's format table and length rule (CPU only).

Each pin checks the oracle against a statement on the pages other than the
one the oracle's table was typed from: the NInfer GGUF table, the ONNX field
layouts (byte sums), the bits/weight columns and the gld-kiln group count.
"""
import re
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden

TYPE_BYTES = {"h": 2, "f": 4, "u8": 1, "i8": 1, "u16": 2, "i16": 2}


def test_table_matches_onnx_quantization_formats(orc):
    rows = read_golden("gguf_block_table.txt")
    assert len(rows) == 27
    for ident, B, S in rows:
        b, s, _ = orc.format_info(ident)
        assert (b, s) == (int(B), int(S)), ident
    gguf_in_oracle = [f for f in orc.formats() if f.startswith("gguf:")]
    assert sorted(gguf_in_oracle) == sorted(r[0] for r in rows)


def test_table_matches_ninfer_gguf_table(orc):
    # The NInfer table is a second, independent statement of (B, S); its
    # bits/weight column must equal 8*S/B.
    for name, _ggml_type, B, S, bpw in read_golden("ninfer_gguf_table.txt"):
        ident = "gguf:" + name[len("gguf_"):]
        b, s, _ = orc.format_info(ident)
        assert (b, s) == (int(B), int(S)), ident
        assert Fraction(8 * s, b) == Fraction(bpw), ident


def test_block_bytes_equal_field_byte_sums(orc):
    for fmt, *fields in read_golden("field_layouts.txt"):
        total = 0
        for tok in fields:
            m = re.fullmatch(r"(\w+):(\w+)(?:\[(\d+)\])?", tok)
            assert m, tok
            total += TYPE_BYTES[m.group(1)] * int(m.group(3) or 1)
        _, s, _ = orc.format_info("gguf:" + fmt.lower())
        assert s == total, fmt


def test_grouped_format_readings_match_bits_per_weight(orc):
    # The byte layouts of q4_g64_fp16 / q8_g32_fp16 are readings; their cost
    # per weight must still be b + 16/G as the NInfer grouped table states.
    rows = {r[0]: r for r in read_golden("ninfer_grouped_table.txt")}
    for name in ("q4_g64_fp16", "q8_g32_fp16"):
        _, b, G, _, _, bpw = rows[name]
        B, S, dec = orc.format_info(name)
        assert dec and B == int(G)
        assert Fraction(int(b)) + Fraction(16, int(G)) == Fraction(bpw)
        assert Fraction(8 * S, B) == Fraction(bpw)


def test_decoded_set(orc):
    decoded = {f for f in orc.formats() if orc.format_info(f)[2]}
    assert decoded == {"gguf:q8_0", "gguf:q4_0", "gguf:q4_k", "gguf:q6_k", "gguf:iq4_nl",
                       "gguf:mxfp4", "gguf:nvfp4", "nvfp4", "q4_g64_fp16", "q8_g32_fp16",
                       "gguf:q4_1", "gguf:q5_0", "gguf:q5_1", "gguf:q8_1", "gguf:q8_k", "gguf:q2_k",
                       "gguf:q3_k", "gguf:q5_k", "gguf:iq4_xs", "gguf:tq1_0", "gguf:tq2_0", "gguf:q1_0",
                       "gguf:q2_0", "gguf:iq2_xxs", "gguf:iq2_xs", "gguf:iq2_s", "gguf:iq3_xxs", "gguf:iq3_s",
                       "gguf:iq1_s", "gguf:iq1_m", "q2_g64_fp16", "q5_g64_fp16", "q6_g64_fp16", "t2_g128_fp16",
                       "fp8_e4m3fn_row_bf16", "fp8_e4m3fn_row_fp16"}
    assert decoded == set(orc.formats())


@pytest.mark.parametrize("fmt,shape", [
    ("gguf:q8_0", (256, 4096)), ("gguf:q4_0", (4096, 4096)), ("q4_g64_fp16", (4096, 4096)),
    ("gguf:q4_k", (14336, 4096)), ("gguf:q6_k", (14336, 4096)), ("gguf:mxfp4", (8192, 28672)),
    ("gguf:iq4_nl", (8192, 28672)), ("gguf:q8_0", (128256, 4096)), ("gguf:q4_k", (2, 3, 512)),
    ("gguf:q8_0", (32,)),
])
def test_block_count_equals_kiln_group_count(orc, fmt, shape):
    B, S, _ = orc.format_info(fmt)
    groups = orc.kiln_group_count(shape, len(shape) - 1, B)
    nb, rows, _ = orc.geometry(fmt, shape, groups * S)
    assert nb == groups


def test_kiln_worked_example(orc):
    rows = read_golden("kiln_examples.txt")
    shape, axis, g, count = rows[0]
    shp = tuple(int(s) for s in shape.split(","))
    assert orc.kiln_group_count(shp, int(axis), int(g)) == int(count)
    # The same example is one MXFP4 block: 32 elements, one e8m0 byte.
    nb, _, _ = orc.geometry("gguf:mxfp4", shp, 17)
    assert nb == 1


def test_length_rule_errors(orc):
    E = orc.OracleError
    with pytest.raises(E) as e:
        orc.geometry("gguf:q4_0", (4, 33), 4 * 18)
    assert e.value.name == "not_block_aligned"
    with pytest.raises(E) as e:
        orc.geometry("gguf:q4_0", (4, 32), 4 * 18 + 1)
    assert e.value.name == "length_mismatch"
    with pytest.raises(E) as e:
        orc.geometry("gguf:q4_0", (-1, 32), 0)
    assert e.value.name == "negative_dim"
    with pytest.raises(E) as e:
        orc.geometry("gguf:q4_0", (), 0)
    assert e.value.name == "bad_rank"
    with pytest.raises(E) as e:
        orc.geometry("gguf:Q4_0", (1, 32), 18)  # case-sensitive identifiers
    assert e.value.name == "unknown_format"
    with pytest.raises(E) as e:
        orc.geometry("gguf:q4_0(32)", (1, 32), 18)  # parameterised spelling
    assert e.value.name == "unknown_format"
    with pytest.raises(E) as e:
        orc.geometry("gguf:q8_0", (2**40, 2**40, 32), 0)
    assert e.value.name == "overflow"


def test_empty_tensors(orc):
    # A zero dimension gives an empty output; the last dim stays block-aligned.
    assert orc.geometry("gguf:q4_k", (0, 256), 0)[0] == 0
    assert orc.geometry("gguf:q4_k", (7, 0), 0)[0] == 0
    with pytest.raises(orc.OracleError):
        orc.geometry("gguf:q4_k", (0, 100), 0)
    y = orc.decode("gguf:q4_k", (0, 256), np.zeros(0, np.uint8), "bfloat16")
    assert y.shape == (0, 256)


def test_nvfp4_divisor_geometry(orc):
    # READING: D >= 1 FP32 divisors follow the blocks; D divides the row count.
    nb = 6 * (128 // 64)
    assert orc.geometry("nvfp4", (6, 128), nb * 36 + 4)[2] == 1
    assert orc.geometry("nvfp4", (6, 128), nb * 36 + 12)[2] == 3
    for bad in (nb * 36, nb * 36 + 2, nb * 36 + 16):  # D=0, ragged, D=4 (4 does not divide 6)
        with pytest.raises(orc.OracleError):
            orc.geometry("nvfp4", (6, 128), bad)
