"""The oracle's pins catch planted mistakes.

Each mutant below is a copy of the oracle's C source with one plausible
mistake, in the shared helpers or in one format's decoder: a wrong
exponent bias or scale, a wrong table entry, a transposed loop or bit
order, a wrong index, offset or sign, a dropped term or parity, a rounding
tie broken the wrong way, a reciprocal multiply in place of a division, a
dropped validation rule.  For each, the oracle's own pin tests (tables, scalars,
formats and the other families) run against the mutant in a subprocess and
must fail.  CPU only: the mistakes are planted in the oracle, never in the
CUDA library.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ndq_oracle.c")
PIN_TESTS = ["tests/test_oracle_tables.py", "tests/test_oracle_scalars.py", "tests/test_oracle_formats.py",
             "tests/test_oracle_next.py", "tests/test_oracle_grouped_fp8.py", "tests/test_oracle_iq.py",
             "tests/test_oracle_matmul.py"]

# (name, text in the oracle, replacement): one mistake each
MUTANTS = [
    ("binary16 exponent bias", "((e - 15u + 127u) << 23)", "((e - 14u + 127u) << 23)"),
    ("binary16 subnormal scale", "ldexpf((float)m, -24)", "ldexpf((float)m, -25)"),
    ("E8M0 half scale below 2", "(0x00200000u << e)", "(0x00400000u << e)"),
    ("unsigned-E4M3 byte 127 not zero", "if (e == 0 || e == 127) return 0.0f;", "if (e == 0) return 0.0f;"),
    ("E4M3FN NaN word", "if (e == 15u && m == 7u)", "if (e == 15u && m == 6u)"),
    ("E4M3FN subnormal scale", "v = ldexpf((float)m, -9);", "v = ldexpf((float)m, -10);"),
    ("E2M1 value 6", "4.0f, 6.0f};", "4.0f, 5.0f};"),
    ("doubled E2M1 table entry", "-6, -8, -12};", "-6, -8, -11};"),
    ("IQ4_NL table entry", "25,  38,", "25,  37,"),
    ("bfloat16 ties away from zero", "u += 0x7fffu + lsb;", "u += 0x8000u + 0u * lsb;"),
    ("binary16 overflow threshold", "if (a >= 0x477ff000u)", "if (a >= 0x477fe000u)"),
    ("plane order transposed",
     "        for (int p = 0; p < 8 / w; ++p)\n            for (int j = 0; j < g; ++j) out[n++]",
     "        for (int j = 0; j < g; ++j)\n            for (int p = 0; p < 8 / w; ++p) out[n++]"),
    ("q8_0 codes unsigned", "M(d, (float)signed8(b[2 + j]))", "M(d, (float)b[2 + j])"),
    ("q4_0 offset", "y[j] = M(d, (float)((int32_t)v[j] - 8));", "y[j] = M(d, (float)((int32_t)v[j] - 7));"),
    ("q4_k high scale bits from the wrong byte", "a[k] = (s[k + 4] % 16u) + 16u * (uint32_t)(s[k - 4] / 64u);",
     "a[k] = (s[k + 4] % 16u) + 16u * (uint32_t)(s[k] / 64u);"),
    ("q5_k high min bits from the wrong byte", "*m = (uint32_t)(s[k + 4] / 16u) + 16u * (uint32_t)(s[k] / 64u);",
     "*m = (uint32_t)(s[k + 4] / 16u) + 16u * (uint32_t)(s[k - 4] / 64u);"),
    ("q4_k min added", "D(M(M(d, (float)a[k]), (float)v[j]), M(dmin, (float)m[k]))",
     "A(M(M(d, (float)a[k]), (float)v[j]), M(dmin, (float)m[k]))"),
    ("q6_k offset", "16 * (int32_t)h[j] - 32;", "16 * (int32_t)h[j] - 31;"),
    ("q6_k scale index", "signed8(b[192 + j / 16])", "signed8(b[192 + j / 32])"),
    ("nvfp4 reciprocal multiply", "y[16 * g + j] = prod / dw;", "y[16 * g + j] = prod * (1.0f / dw);"),
    ("q4_g64 two's complement", "(int32_t)u - 16;", "(int32_t)u - 15;"),
    ("length rule: last dimension not checked", "if (K % B != 0) return OR_ERR_NOT_BLOCK_ALIGNED;",
     "if (0) return OR_ERR_NOT_BLOCK_ALIGNED;"),
    ("nvfp4 divisor count must divide the rows", "if (D < 1 || N % D != 0) return OR_ERR_LENGTH_MISMATCH;",
     "if (D < 1) return OR_ERR_LENGTH_MISMATCH;"),
    # the other gguf formats
    ("q4_1 minimum subtracted", "y[j] = A(M(d, (float)v[j]), m);", "y[j] = D(M(d, (float)v[j]), m);"),
    ("q5_0 offset", "M(d, (float)((int32_t)vj - 16))", "M(d, (float)((int32_t)vj - 15))"),
    ("q5 high bits in the wrong order", "16u * ((high >> j) & 1u)", "16u * ((high >> (j ^ 1)) & 1u)"),
    ("q8_1 codes read over the cached sum", "for (int j = 0; j < 32; ++j) y[j] = M(d, (float)signed8(b[4 + j]));",
     "for (int j = 0; j < 32; ++j) y[j] = M(d, (float)signed8(b[2 + j]));"),
    ("q8_k scale read as binary16", "float d = or_f32(U(b, 4));", "float d = H(b);"),
    ("q2_k minimum from the low nibble", "M(dmin, (float)(sc / 16u))", "M(dmin, (float)(sc % 16u))"),
    ("q3_k mask sense", "4 * (1 - (int32_t)h[j])", "4 * (int32_t)h[j]"),
    ("q5_k high bit weight", "(float)(v[j] + 16u * hb[j])", "(float)(v[j] + 8u * hb[j])"),
    ("iq4_xs scale offset", "16 * (int32_t)field(high, 2 * k, 2) - 32;", "16 * (int32_t)field(high, 2 * k, 2) - 31;"),
    ("tq1_0 trit divisor", "(int32_t)((3u * r) / 256u) - 1", "(int32_t)((3u * r) / 255u) - 1"),
    ("tq2_0 offset", "for (int j = 0; j < 256; ++j) y[j] = M(d, (float)((int32_t)v[j] - 1));",
     "for (int j = 0; j < 256; ++j) y[j] = M(d, (float)((int32_t)v[j] - 2));"),
    ("q1_0 bit sense", "? d : -d;", "? -d : d;"),
    ("q2_0 plane grouping", "P(b + 2, 16, 2, 1, v);", "P(b + 2, 16, 2, 16, v);"),
    # the IQ formats
    ("IQ sign parity dropped", "S8((v & 127u) | ((par % 2u) << 7), s);", "S8((v & 127u) | (0u * par), s);"),
    ("iq2_xxs scale factor", "A(0.5f, (float)(a >> 28))), 0.25f)", "A(0.5f, (float)(a >> 28))), 0.125f)"),
    ("iq3_s odd multiplier", "(float)(1u + 2u * field(b[106 + g / 2], 4 * (g % 2), 4))",
     "(float)(2u * field(b[106 + g / 2], 4 * (g % 2), 4))"),
    ("iq1_s shift sign", "float delta = field(a, 15, 1) ? -0.125f : 0.125f;",
     "float delta = field(a, 15, 1) ? 0.125f : -0.125f;"),
    ("iq1_m scale nibble order", "dbits += (w[k] >> 12) << (4 * k);", "dbits += (w[k] >> 12) << (4 * (3 - k));"),
    # the other NInfer formats
    ("grouped two's complement range", "(int32_t)u - (int32_t)(1u << width)",
     "(int32_t)u - (int32_t)(1u << (width - 1))"),
    ("grouped bit stream order", "v |= (uint32_t)field(a[bitpos / 8], bitpos % 8, 1) << t;",
     "v |= (uint32_t)field(a[bitpos / 8], bitpos % 8, 1) << (width - 1 - t);"),
    ("q2_g64 grid offset", "or_stream_word(b + 2, k, 2) - 1", "or_stream_word(b + 2, k, 2) - 2"),
    ("fp8 row multiplier dropped", "y[0] = M(oracle_e4m3fn(b[0]), s32);", "y[0] = oracle_e4m3fn(b[0]) + 0.0f * s32;"),
    ("BF16 multiplier bits", "or_f32(w << 16)", "or_f32(w << 15)"),
    # the fused-product reference
    ("product activation index transposed", "or_bf16_to_f64(x_bf16[m * K + k]) * (double)row[k]",
     "or_bf16_to_f64(x_bf16[k * M + m]) * (double)row[k]"),
    ("product output index transposed", "y[m * N + n] = s;", "y[n * M + m] = s;"),
    ("product weight row offset", "w, w_len, n * bpr, (n + 1) * bpr, row);", "w, w_len, n * K, n * K + bpr, row);"),
    ("product bfloat16 weights not rounded", "if (weight_dtype == 2) /* bfloat16 bit patterns",
     "if (weight_dtype == 3) /* bfloat16 bit patterns"),
]


def _run_pins(name, find, repl, tmp):
    src = open(SRC).read()
    assert src.count(find) == 1, f"{name}: the text to mutate must occur once"
    d = os.path.join(tmp, name.replace(" ", "_").replace("'", "").replace(":", ""))
    os.makedirs(d)
    msrc = os.path.join(d, "ndq_oracle.c")
    with open(msrc, "w") as f:
        f.write(src.replace(find, repl))
    lib = os.path.join(d, "liboracle.so")
    # the mutant must compile: a build failure would "kill" it for nothing
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-o", lib,
                    msrc, "-lm"], check=True, capture_output=True)
    env = dict(os.environ, NDQ_ORACLE_SRC=msrc, NDQ_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
                        *PIN_TESTS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    return name, r.returncode, r.stdout[-600:]


def test_pins_kill_every_mutant(tmp_path):
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda m: _run_pins(*m, str(tmp_path)), MUTANTS))
    survivors = [(name, out) for name, rc, out in results if rc == 0]
    assert not survivors, "mutants the pins did not catch: " + "; ".join(n for n, _ in survivors)
    # a killed mutant fails a test; it does not break the collection
    for name, rc, out in results:
        assert rc == 1, f"{name}: pytest exit code {rc}\n{out}"


def test_unmutated_oracle_passes_the_pins():
    # the same subprocess harness on the real oracle passes (so a failing
    # mutant run is due to its mistake)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
                        *PIN_TESTS], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutation_text_occurs_once(name, find, repl):
    assert open(SRC).read().count(find) == 1, name
    assert find != repl
