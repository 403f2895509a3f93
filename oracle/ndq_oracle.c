/*
 * ndq_oracle.c -- plain, slow, single-threaded CPU decoder of packed quantized
 * weight payloads.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity reference that the CUDA
 * library is checked against and the timed CPU baseline.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg load it.  It shares no
 * source, header, table or helper with the CUDA library
 * (quantized_weight_block_gb300/csrc); the two agree only because both follow
 * the same published definitions.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * -ffp-contract=off is required: every M/A/D below must round separately
 * to binary32 ("ONNX DequantizePacked decoding specification", section
 * "Decoding algorithms": each addition, subtraction and multiplication is
 * rounded independently; nested calls are not fused or reassociated).
 *
 * Sources (page title, section):
 *  [DQP]   ONNX "DequantizePacked decoding specification" (opset 29):
 *          "Signature and storage", "Quantization formats" (B,S table),
 *          "Packed layouts and decoding" (field table),
 *          "Mathematical decoding rules" (P, M/A/D and per-format rules).
 *  [NINF]  NInfer "tensor-formats" maintainer reference: section 3.3 (nvfp4,
 *          E2M1, E4M3FN, divisor), sections 4-6.2 (grouped signed-integer
 *          schemes and their binary32 reconstruction), section 7.2
 *          (grouped_absmax canonical encoder), GGUF block table.
 *  [KILN]  gld-kiln "Quantization" spec: group-count formula, E8M0 byte 127.
 *
 * The IQ codebooks ([DQP] "IQ codebooks") are page data; the test harness
 * passes them in from a cited text fixture (oracle_set_codebook) and the
 * IQ decoders report an unsupported format until they are loaded.
 *
 * Readings where the pages leave a step open are marked READING and listed
 * in the design notes.
 *
 * Parity pins: every function here is pinned by a CPU test against something
 * other than itself (library routines, closed forms, exhaustive enumerations,
 * hand-built blocks with known values, exact-rational evaluation, encoder
 * round trips).  "parity unpinned": none of the decode functions; the upstream
 * ggml digest corpus named by the pages is not available, so agreement with
 * ggml's own C decoders is not checked.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_NULL 1
#define OR_ERR_UNKNOWN_FORMAT 2
#define OR_ERR_UNSUPPORTED_FORMAT 3
#define OR_ERR_BAD_RANK 4
#define OR_ERR_NEGATIVE_DIM 5
#define OR_ERR_NOT_BLOCK_ALIGNED 6
#define OR_ERR_LENGTH_MISMATCH 7
#define OR_ERR_OVERFLOW 8
#define OR_ERR_BAD_DTYPE 9
#define OR_ERR_RANGE 10
#define OR_ERR_ENCODE 11

/* ------------------------------------------------------------------------ */
/* Format registry.                                                          */
/* [DQP] "Quantization formats": the 27 fixed GGUF profiles with their       */
/* decoded element count B and packed byte count S.  The last three rows are */
/* [NINF] formats; their byte layout is a READING (see oracle_format_info).  */
/* ------------------------------------------------------------------------ */
typedef struct {
    const char *name;
    int B;
    int S;
    int decoded; /* 1 if this oracle decodes it */
} or_format;

static const or_format OR_FORMATS[] = {
    {"gguf:q4_0", 32, 18, 1},     {"gguf:q4_1", 32, 20, 1},
    {"gguf:q5_0", 32, 22, 1},     {"gguf:q5_1", 32, 24, 1},
    {"gguf:q8_0", 32, 34, 1},     {"gguf:q8_1", 32, 36, 1},
    {"gguf:q2_k", 256, 84, 1},    {"gguf:q3_k", 256, 110, 1},
    {"gguf:q4_k", 256, 144, 1},   {"gguf:q5_k", 256, 176, 1},
    {"gguf:q6_k", 256, 210, 1},   {"gguf:q8_k", 256, 292, 1},
    {"gguf:iq2_xxs", 256, 66, 1}, {"gguf:iq2_xs", 256, 74, 1},
    {"gguf:iq3_xxs", 256, 98, 1}, {"gguf:iq1_s", 256, 50, 1},
    {"gguf:iq4_nl", 32, 18, 1},   {"gguf:iq3_s", 256, 110, 1},
    {"gguf:iq2_s", 256, 82, 1},   {"gguf:iq4_xs", 256, 136, 1},
    {"gguf:iq1_m", 256, 56, 1},   {"gguf:tq1_0", 256, 54, 1},
    {"gguf:tq2_0", 256, 66, 1},   {"gguf:mxfp4", 32, 17, 1},
    {"gguf:nvfp4", 64, 36, 1},    {"gguf:q1_0", 128, 18, 1},
    {"gguf:q2_0", 64, 18, 1},
    /* [NINF] formats.  READING: nvfp4 uses the gguf:nvfp4 block geometry
     * (4 scale bytes then 32 code bytes per 64 values) and appends its FP32
     * divisors after the last block; q4_g64_fp16 is one binary16 scale then
     * 32 bytes of adjacent two's-complement nibbles; q8_g32_fp16 is one
     * binary16 scale then 32 signed bytes. */
    {"nvfp4", 64, 36, 1},
    {"q4_g64_fp16", 64, 34, 1},
    {"q8_g32_fp16", 32, 34, 1},
    /* READING: q2/q5/q6_g64_fp16 and t2_g128_fp16 follow q4_g64_fp16: one
     * binary16 scale, then the group's codes as an LSB-first bit stream
     * (S = 2 + G*b/8).  The row-scaled FP8 formats are a code plane of
     * N*K E4M3FN bytes (row-major) followed by a plane of N little-endian
     * 16-bit row multipliers; a "block" is one code (B = S = 1). */
    {"q2_g64_fp16", 64, 18, 1},
    {"q5_g64_fp16", 64, 42, 1},
    {"q6_g64_fp16", 64, 50, 1},
    {"t2_g128_fp16", 128, 34, 1},
    {"fp8_e4m3fn_row_bf16", 1, 1, 1},
    {"fp8_e4m3fn_row_fp16", 1, 1, 1},
};
#define OR_NFORMATS ((int)(sizeof(OR_FORMATS) / sizeof(OR_FORMATS[0])))

/* Case-sensitive exact match; parameterised spellings are simply unknown
 * ([DQP] "Format identifiers"). */
static int or_find(const char *name) {
    if (!name) return -1;
    for (int i = 0; i < OR_NFORMATS; ++i)
        if (strcmp(OR_FORMATS[i].name, name) == 0) return i;
    return -1;
}

int oracle_format_count(void) { return OR_NFORMATS; }

const char *oracle_format_name(int i) {
    return (i >= 0 && i < OR_NFORMATS) ? OR_FORMATS[i].name : NULL;
}

int oracle_format_info(const char *name, int *B, int *S, int *decoded) {
    int i = or_find(name);
    if (i < 0) return OR_ERR_UNKNOWN_FORMAT;
    if (B) *B = OR_FORMATS[i].B;
    if (S) *S = OR_FORMATS[i].S;
    if (decoded) *decoded = OR_FORMATS[i].decoded;
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Scalar building blocks.                                                   */
/* ------------------------------------------------------------------------ */
static float or_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t or_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* M, A, D of [DQP] "Mathematical decoding rules": one binary32 RNE rounding
 * each.  Kept as functions so that no expression below can be contracted. */
static inline float M(float a, float b) { return a * b; }
static inline float A(float a, float b) { return a + b; }
static inline float D(float a, float b) { return a - b; }

/* Unsigned little-endian integer of `count` bytes ([DQP] U(a)). */
static uint32_t U(const uint8_t *a, int count) {
    uint32_t v = 0;
    for (int j = 0; j < count; ++j) v |= (uint32_t)a[j] << (8 * j);
    return v;
}

/* field(v,k,w) = floor(v / 2^k) mod 2^w   ([DQP] "Mathematical decoding rules") */
static uint32_t field(uint32_t v, int k, int w) { return (v >> k) & ((1u << w) - 1u); }

/* Exact binary16 -> binary32 ([DQP] H; IEEE 754 binary16: 1 sign bit, 5
 * exponent bits with bias 15, 10 fraction bits).  Built from the bit
 * pattern so that no arithmetic rounding can enter. */
float oracle_h2f(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t e = (h >> 10) & 31u;
    uint32_t m = h & 1023u;
    if (e == 31u) /* infinity (m == 0) or NaN (payload kept) */
        return or_f32(sign | 0x7f800000u | (m << 13));
    if (e == 0u) {
        if (m == 0u) return or_f32(sign); /* signed zero */
        /* subnormal: m * 2^-24, exact in binary32 */
        float v = ldexpf((float)m, -24);
        return sign ? -v : v;
    }
    return or_f32(sign | ((e - 15u + 127u) << 23) | (m << 13));
}

static float H(const uint8_t *p) { return oracle_h2f((uint16_t)U(p, 2)); }

/* MXFP4 half scale ([DQP] "Ternary and block-floating formats"): the FLOAT
 * whose bit pattern is 0x00200000 * 2^e for e < 2, and (e-1) * 2^23
 * otherwise.  Byte 127 gives 2^-1, i.e. a block scale of exactly 1.0 once
 * applied to the doubled E2M1 table ([KILN]: e8m0 byte 127 is the MXFP4
 * block of 32 at unit scale). */
float oracle_e8m0_half(uint8_t e) {
    uint32_t bits = (e < 2) ? (0x00200000u << e) : ((uint32_t)(e - 1) << 23);
    return or_f32(bits);
}

/* gguf:nvfp4 unsigned E4M3 half scale ([DQP] "Ternary and block-floating
 * formats", NVFP4): zero when the whole byte is 0 or 127; otherwise with
 * E = field(e,3,4) and m = e mod 8, m * 2^-10 if E == 0 else
 * (1 + m/8) * 2^(E-8).  Bit 7 enters neither E nor m. */
float oracle_ue4m3_half(uint8_t e) {
    if (e == 0 || e == 127) return 0.0f;
    uint32_t E = field(e, 3, 4), m = e % 8u;
    if (E == 0) return ldexpf((float)m, -10);
    return ldexpf((float)(8u + m), (int)E - 8 - 3); /* (1+m/8)*2^(E-8) */
}

/* E4M3FN word ([NINF] section 3.3): sign bit 7, exponent bits 6:3, fraction
 * bits 2:0, bias 7.  e=0,m=0 signed zero; e=0 subnormal m*2^-9;
 * 1<=e<=14 normal; e=15,m<7 normal (1+m/8)*2^8; e=15,m=7 NaN. */
float oracle_e4m3fn(uint8_t w) {
    int neg = (w >> 7) & 1;
    uint32_t e = field(w, 3, 4), m = w & 7u;
    float v;
    if (e == 15u && m == 7u) {
        v = or_f32(0x7fc00000u);
    } else if (e == 0u) {
        v = ldexpf((float)m, -9); /* m == 0 gives +0, sign applied below */
    } else {
        v = ldexpf((float)(8u + m), (int)e - 7 - 3);
    }
    return neg ? -v : v;
}

/* E2M1 word ([NINF] section 3.3): positive words 0..7 are 0, 0.5, 1, 1.5, 2,
 * 3, 4, 6; bit 3 negates, so 0x8 is negative zero. */
float oracle_e2m1(uint8_t c) {
    static const float pos[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    float v = pos[c & 7u];
    return (c & 8u) ? -v : v;
}

/* Doubled E2M1 table used with a half scale by gguf:mxfp4 and gguf:nvfp4
 * ([DQP] "Ternary and block-floating formats"); both zero entries are +0. */
static const float OR_V[16] = {0, 1, 2, 3, 4, 6, 8, 12, 0, -1, -2, -3, -4, -6, -8, -12};

/* IQ4_NL 16-entry nonlinear table ([DQP] "Packed layouts and decoding"). */
static const int OR_IQ4[16] = {-127, -104, -83, -65, -49, -35, -22, -10,
                               1,    13,   25,  38,  53,  69,  89,  113};

/* Output casts ([DQP] "Signature and storage": FLOAT16 and BFLOAT16 by
 * round-to-nearest, ties-to-even).  Integer rounding on the binary32 bit
 * pattern; NaN stays NaN (quieted, sign kept); overflow rounds to infinity;
 * subnormals and signed zeros are kept (no flush). */
uint16_t oracle_f32_to_bf16(uint32_t u) {
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

uint16_t oracle_f32_to_f16(uint32_t u) {
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return (uint16_t)(sign | 0x7e00u | ((a >> 13) & 0x3ffu));
    if (a >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u); /* >= 65520 rounds to inf */
    if (a >= 0x38800000u) {                                  /* binary16 normal range */
        uint32_t h = (a >> 13) - ((127u - 15u) << 10);
        uint32_t rem = a & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
        return (uint16_t)(sign | h);
    }
    /* binary16 subnormal or zero: value in units of 2^-24 */
    uint32_t e = a >> 23;
    uint64_t m = (e == 0u) ? (a & 0x7fffffu) : ((a & 0x7fffffu) | 0x800000u);
    int shift = (e == 0u) ? 125 : (int)(126u - e); /* m * 2^(e-150) / 2^-24 */
    if (shift >= 40) return sign;
    uint64_t q = m >> shift;
    uint64_t rem = m & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1ull))) q += 1ull;
    return (uint16_t)(sign | (uint16_t)q);
}

/* P(a,w,g) of [DQP] "Mathematical decoding rules": field(a[s+j], w*p, w)
 * enumerated over byte-group starts s = 0,g,2g,...; then bit planes
 * p = 0..8/w-1; then bytes j = 0..g-1.  Writes len*8/w values. */
static void P(const uint8_t *a, int len, int w, int g, uint32_t *out) {
    int n = 0;
    for (int s = 0; s < len; s += g)
        for (int p = 0; p < 8 / w; ++p)
            for (int j = 0; j < g; ++j) out[n++] = field(a[s + j], w * p, w);
}

static int32_t signed8(uint8_t v) { return (v & 128u) ? (int32_t)v - 256 : (int32_t)v; }

/* ------------------------------------------------------------------------ */
/* Per-block decoders: one block of S bytes -> B binary32 values, in the     */
/* pages' operation order.                                                   */
/* ------------------------------------------------------------------------ */

/* gguf:q8_0 and q8_g32_fp16.  [DQP] Q8_0: fields h d; i8 q[32];
 * y[j] = M(d, q[j]).  [NINF] section 6.2: w = binary32(s32 * binary32(q)),
 * the same product for the READING that q8_g32_fp16 stores one binary16
 * scale followed by 32 signed bytes. */
static void dec_q8_0(const uint8_t *b, float *y) {
    float d = H(b);
    for (int j = 0; j < 32; ++j) y[j] = M(d, (float)signed8(b[2 + j]));
}

/* gguf:q4_0.  Fields h d; u8 q[16].  v = P(q,4,16); y[j] = M(d, v[j]-8). */
static void dec_q4_0(const uint8_t *b, float *y) {
    uint32_t v[32];
    float d = H(b);
    P(b + 2, 16, 4, 16, v);
    for (int j = 0; j < 32; ++j) y[j] = M(d, (float)((int32_t)v[j] - 8));
}

/* gguf:iq4_nl.  Fields h d; u8 q[16].  v = P(q,4,16); y[j] = M(d, IQ4[v[j]]). */
static void dec_iq4_nl(const uint8_t *b, float *y) {
    uint32_t v[32];
    float d = H(b);
    P(b + 2, 16, 4, 16, v);
    for (int j = 0; j < 32; ++j) y[j] = M(d, (float)OR_IQ4[v[j]]);
}

/* gguf:q4_k.  Fields h d; h dmin; u8 scales[12]; u8 q[128].  v = P(q,4,32);
 * 6-bit a[k], m[k] unpacked from the 12 scale bytes s:
 *   k < 4 : a = s[k] mod 64, m = s[k+4] mod 64
 *   k >= 4: a = (s[k+4] mod 16) + 16*floor(s[k-4]/64),
 *           m = floor(s[k+4]/16) + 16*floor(s[k]/64)
 * y[j] = D(M(M(d, a[k]), v[j]), M(dmin, m[k])) with k = floor(j/32). */
static void dec_q4_k(const uint8_t *b, float *y) {
    uint32_t v[256], a[8], m[8];
    const uint8_t *s = b + 4;
    float d = H(b), dmin = H(b + 2);
    for (int k = 0; k < 8; ++k) {
        if (k < 4) {
            a[k] = s[k] % 64u;
            m[k] = s[k + 4] % 64u;
        } else {
            a[k] = (s[k + 4] % 16u) + 16u * (uint32_t)(s[k - 4] / 64u);
            m[k] = (uint32_t)(s[k + 4] / 16u) + 16u * (uint32_t)(s[k] / 64u);
        }
    }
    P(b + 16, 128, 4, 32, v);
    for (int j = 0; j < 256; ++j) {
        int k = j / 32;
        y[j] = D(M(M(d, (float)a[k]), (float)v[j]), M(dmin, (float)m[k]));
    }
}

/* gguf:q6_k.  Fields u8 low[128]; u8 high[64]; i8 scales[16]; h d.
 * l = P(low,4,64), h = P(high,2,32), s = scales[floor(j/16)] signed;
 * y[j] = M(M(d, s), l[j] + 16*h[j] - 32). */
static void dec_q6_k(const uint8_t *b, float *y) {
    uint32_t l[256], h[256];
    float d = H(b + 208);
    P(b, 128, 4, 64, l);
    P(b + 128, 64, 2, 32, h);
    for (int j = 0; j < 256; ++j) {
        int32_t s = signed8(b[192 + j / 16]);
        int32_t q = (int32_t)l[j] + 16 * (int32_t)h[j] - 32;
        y[j] = M(M(d, (float)s), (float)q);
    }
}

/* gguf:mxfp4.  Fields u8 exponent; u8 q[16].  d = half scale of the
 * exponent byte; v = P(q,4,16); y[j] = M(d, V[v[j]]). */
static void dec_mxfp4(const uint8_t *b, float *y) {
    uint32_t v[32];
    float d = oracle_e8m0_half(b[0]);
    P(b + 1, 16, 4, 16, v);
    for (int j = 0; j < 32; ++j) y[j] = M(d, OR_V[v[j]]);
}

/* gguf:nvfp4.  Fields u8 scales[4]; u8 q[32]: four groups of 16.  For group
 * g: d = unsigned-E4M3 half scale of scales[g]; v = P(q[8g:8g+8],4,8);
 * y[16g+j] = M(d, V[v[j]]). */
static void dec_gguf_nvfp4(const uint8_t *b, float *y) {
    uint32_t v[16];
    for (int g = 0; g < 4; ++g) {
        float d = oracle_ue4m3_half(b[g]);
        P(b + 4 + 8 * g, 8, 4, 8, v);
        for (int j = 0; j < 16; ++j) y[16 * g + j] = M(d, OR_V[v[j]]);
    }
}

/* nvfp4 ([NINF] section 3.3):
 *   W = decode_e2m1(c) * decode_e4m3fn(s) / d_w
 * READING: the product is formed first (it is exact in binary32) and the
 * quotient is rounded once to binary32, round-to-nearest-even (IEEE
 * division).  Block geometry as gguf:nvfp4: scale byte g covers elements
 * 16g..16g+15 of the block, codes in P(q[8g:8g+8],4,8) order. */
static void dec_nvfp4(const uint8_t *b, float dw, float *y) {
    uint32_t v[16];
    for (int g = 0; g < 4; ++g) {
        float s = oracle_e4m3fn(b[g]);
        P(b + 4 + 8 * g, 8, 4, 8, v);
        for (int j = 0; j < 16; ++j) {
            float prod = M(oracle_e2m1((uint8_t)v[j]), s);
            y[16 * g + j] = prod / dw;
        }
    }
}

/* q4_g64_fp16 ([NINF] sections 5-6.2): 4-bit two's-complement code
 * q = u if u < 8 else u - 16; w = binary32(s32 * binary32(q)).  The scale
 * is a signed multiplier.  READING of the byte layout: binary16 scale at
 * offset 0, then element k in bits 4*(k mod 2) of byte 2 + floor(k/2). */
static void dec_q4_g64(const uint8_t *b, float *y) {
    float s32 = H(b);
    for (int k = 0; k < 64; ++k) {
        uint32_t u = field(b[2 + k / 2], 4 * (k % 2), 4);
        int32_t q = (u < 8u) ? (int32_t)u : (int32_t)u - 16;
        y[k] = M(s32, (float)q);
    }
}

/* gguf:q4_1.  Fields h d, m; u8 q[16].  v = P(q,4,16); y[j] = A(M(d,v[j]),m). */
static void dec_q4_1(const uint8_t *b, float *y) {
    uint32_t v[32];
    float d = H(b), m = H(b + 2);
    P(b + 4, 16, 4, 16, v);
    for (int j = 0; j < 32; ++j) y[j] = A(M(d, (float)v[j]), m);
}

/* gguf:q5_0 / q5_1.  Q5_0 fields h d; u8 high[4]; u8 q[16].  Q5_1 fields
 * h d, m; u8 high[4]; u8 q[16].  v = P(q,4,16) with v[j] + 16*bit(U(high),j);
 * Q5_0: y[j] = M(d, v[j]-16); Q5_1: y[j] = A(M(d, v[j]), m). */
static void dec_q5(const uint8_t *b, int affine, float *y) {
    uint32_t v[32];
    int o = affine ? 4 : 2;
    float d = H(b), m = affine ? H(b + 2) : 0.0f;
    uint32_t high = U(b + o, 4);
    P(b + o + 4, 16, 4, 16, v);
    for (int j = 0; j < 32; ++j) {
        uint32_t vj = v[j] + 16u * ((high >> j) & 1u);
        y[j] = affine ? A(M(d, (float)vj), m) : M(d, (float)((int32_t)vj - 16));
    }
}

/* gguf:q8_1 (fields h d, s; i8 q[32]) and gguf:q8_k (fields f d; i8 q[256];
 * i16 sums[16]): y[j] = M(d, q[j]); the cached sum fields are ignored,
 * bits included. */
static void dec_q8_1(const uint8_t *b, float *y) {
    float d = H(b);
    for (int j = 0; j < 32; ++j) y[j] = M(d, (float)signed8(b[4 + j]));
}

static void dec_q8_k(const uint8_t *b, float *y) {
    float d = or_f32(U(b, 4));
    for (int j = 0; j < 256; ++j) y[j] = M(d, (float)signed8(b[4 + j]));
}

/* gguf:q2_k.  Fields u8 scales[16], q[64]; h d, dmin.  v = P(q,2,32),
 * s = scales[floor(j/16)]; y[j] = D(M(M(d, s mod 16), v[j]), M(dmin, floor(s/16))). */
static void dec_q2_k(const uint8_t *b, float *y) {
    uint32_t v[256];
    float d = H(b + 80), dmin = H(b + 82);
    P(b + 16, 64, 2, 32, v);
    for (int j = 0; j < 256; ++j) {
        uint32_t sc = b[j / 16];
        y[j] = D(M(M(d, (float)(sc % 16u)), (float)v[j]), M(dmin, (float)(sc / 16u)));
    }
}

/* gguf:q3_k.  Fields u8 mask[32], q[64], scales[12]; h d.  v = P(q,2,32),
 * h = P(mask,1,32), l = P(b[96:104],4,8), a = P(b[104:108],2,4); with
 * k = floor(j/16) and s = l[k] + 16*a[k] - 32:
 * y[j] = M(M(d, s), v[j] - 4*(1 - h[j])). */
static void dec_q3_k(const uint8_t *b, float *y) {
    uint32_t v[256], h[256], l[16], a[16];
    float d = H(b + 108);
    P(b + 32, 64, 2, 32, v);
    P(b, 32, 1, 32, h);
    P(b + 96, 8, 4, 8, l);
    P(b + 104, 4, 2, 4, a);
    for (int j = 0; j < 256; ++j) {
        int k = j / 16;
        int32_t sc = (int32_t)l[k] + 16 * (int32_t)a[k] - 32;
        int32_t q = (int32_t)v[j] - 4 * (1 - (int32_t)h[j]);
        y[j] = M(M(d, (float)sc), (float)q);
    }
}

/* 6-bit scale a[k] and minimum m[k] of Q4_K / Q5_K from the 12-byte scales
 * field s (see dec_q4_k). */
static void kq_scale_min(const uint8_t *s, int k, uint32_t *a, uint32_t *m) {
    if (k < 4) {
        *a = s[k] % 64u;
        *m = s[k + 4] % 64u;
    } else {
        *a = (s[k + 4] % 16u) + 16u * (uint32_t)(s[k - 4] / 64u);
        *m = (uint32_t)(s[k + 4] / 16u) + 16u * (uint32_t)(s[k] / 64u);
    }
}

/* gguf:q5_k.  Fields h d, dmin; u8 scales[12], high[32], q[128].
 * v = P(q,4,32) + 16*P(high,1,32); a, m as Q4_K;
 * y[j] = D(M(M(d, a[k]), v[j]), M(dmin, m[k])), k = floor(j/32). */
static void dec_q5_k(const uint8_t *b, float *y) {
    uint32_t v[256], hb[256];
    float d = H(b), dmin = H(b + 2);
    P(b + 48, 128, 4, 32, v);
    P(b + 16, 32, 1, 32, hb);
    for (int j = 0; j < 256; ++j) {
        uint32_t a, m;
        kq_scale_min(b + 4, j / 32, &a, &m);
        y[j] = D(M(M(d, (float)a), (float)(v[j] + 16u * hb[j])), M(dmin, (float)m));
    }
}

/* gguf:iq4_xs.  Fields h d; u16 high; u8 scales[4], q[128].  v = P(q,4,16);
 * s[k] = field(scales[floor(k/2)], 4*(k mod 2), 4) + 16*field(high, 2k, 2) - 32;
 * y[j] = M(M(d, s[floor(j/32)]), IQ4[v[j]]). */
static void dec_iq4_xs(const uint8_t *b, float *y) {
    uint32_t v[256];
    float d = H(b);
    uint32_t high = U(b + 2, 2);
    P(b + 8, 128, 4, 16, v);
    for (int j = 0; j < 256; ++j) {
        int k = j / 32;
        int32_t sc = (int32_t)field(b[4 + k / 2], 4 * (k % 2), 4) + 16 * (int32_t)field(high, 2 * k, 2) - 32;
        y[j] = M(M(d, (float)sc), (float)OR_IQ4[v[j]]);
    }
}

/* gguf:tq1_0.  Fields u8 q[48], high[4]; h d.  Three output sequences for
 * (start, width, count) = (0,32,5), (32,16,5), (48,4,4), in that order; in
 * each, p = 0..count-1 before j = 0..width-1; output
 * M(d, floor(3*((b[start+j]*3^p) mod 256)/256) - 1). */
static void dec_tq1_0(const uint8_t *b, float *y) {
    static const int seq[3][3] = {{0, 32, 5}, {32, 16, 5}, {48, 4, 4}};
    float d = H(b + 52);
    int n = 0;
    for (int t = 0; t < 3; ++t) {
        uint32_t pw = 1;
        for (int p = 0; p < seq[t][2]; ++p, pw *= 3u)
            for (int j = 0; j < seq[t][1]; ++j) {
                uint32_t r = (b[seq[t][0] + j] * pw) % 256u;
                int32_t q = (int32_t)((3u * r) / 256u) - 1;
                y[n++] = M(d, (float)q);
            }
    }
}

/* gguf:tq2_0.  Fields u8 q[64]; h d.  y[j] = M(d, v[j]-1), v = P(q,2,32). */
static void dec_tq2_0(const uint8_t *b, float *y) {
    uint32_t v[256];
    float d = H(b + 64);
    P(b, 64, 2, 32, v);
    for (int j = 0; j < 256; ++j) y[j] = M(d, (float)((int32_t)v[j] - 1));
}

/* gguf:q1_0.  Fields h d; u8 q[16].  y[j] = d if bit(q[floor(j/8)], j mod 8)
 * is one, else -d (no multiplication). */
static void dec_q1_0(const uint8_t *b, float *y) {
    float d = H(b);
    for (int j = 0; j < 128; ++j) y[j] = ((b[2 + j / 8] >> (j % 8)) & 1u) ? d : -d;
}

/* gguf:q2_0.  Fields h d; u8 q[16].  y[j] = M(d, v[j]-1), v = P(q,2,1). */
static void dec_q2_0(const uint8_t *b, float *y) {
    uint32_t v[64];
    float d = H(b);
    P(b + 2, 16, 2, 1, v);
    for (int j = 0; j < 64; ++j) y[j] = M(d, (float)((int32_t)v[j] - 1));
}

/* ------------------------------------------------------------------------ */
/* IQ2, IQ3 and IQ1 formats ([DQP] "Mathematical decoding rules", "IQ2,     */
/* IQ3, and IQ1 formats"; tables from [DQP] "IQ codebooks").                 */
/* ------------------------------------------------------------------------ */

/* The six codebooks G(name, r).  Their contents are data printed on the
 * page; the test harness passes each one in as the page's packed bytes
 * (oracle_set_codebook), and this file expands them: entry k is the
 * bits-wide field at bit bits*k of the byte stream (low bits of a byte
 * first) used as an index into the value list, and row r is entries
 * width*r .. width*r + width - 1. */
#define OR_CB_COUNT 6
#define OR_CB_MAX_ENTRIES (2048 * 8)
static const char *const OR_CB_NAMES[OR_CB_COUNT] = {"iq2xxs_grid", "iq2xs_grid", "iq2s_grid",
                                                     "iq3xxs_grid", "iq3s_grid", "iq1s_grid"};
enum { CB_IQ2XXS, CB_IQ2XS, CB_IQ2S, CB_IQ3XXS, CB_IQ3S, CB_IQ1S };
static int8_t OR_CB[OR_CB_COUNT][OR_CB_MAX_ENTRIES];
static int OR_CB_WIDTH[OR_CB_COUNT], OR_CB_ROWS[OR_CB_COUNT];

static int or_cb_find(const char *name) {
    for (int i = 0; i < OR_CB_COUNT; ++i)
        if (name && strcmp(OR_CB_NAMES[i], name) == 0) return i;
    return -1;
}

int oracle_set_codebook(const char *name, int width, int bits, const int32_t *values, int nvalues,
                        const uint8_t *packed, uint64_t nbytes) {
    int ci = or_cb_find(name);
    if (ci < 0) return OR_ERR_UNKNOWN_FORMAT;
    if (!values || !packed) return OR_ERR_NULL;
    if (width < 1 || bits < 1 || bits > 8 || 8 % bits != 0 || nvalues < 1) return OR_ERR_RANGE;
    uint64_t entries = nbytes * 8u / (uint64_t)bits;
    if (entries % (uint64_t)width != 0 || entries > OR_CB_MAX_ENTRIES) return OR_ERR_RANGE;
    for (uint64_t k = 0; k < entries; ++k) {
        uint64_t bit0 = k * (uint64_t)bits;
        uint32_t idx = field(packed[bit0 / 8u], (int)(bit0 % 8u), bits);
        if (idx >= (uint32_t)nvalues) return OR_ERR_RANGE;
        OR_CB[ci][k] = (int8_t)values[idx];
    }
    OR_CB_WIDTH[ci] = width;
    OR_CB_ROWS[ci] = (int)(entries / (uint64_t)width);
    return OR_OK;
}

/* Row r of a loaded codebook into out[0..width-1]; returns the width, or a
 * negative error. */
int oracle_codebook_row(const char *name, int r, int32_t *out) {
    int ci = or_cb_find(name);
    if (ci < 0 || !out) return -OR_ERR_UNKNOWN_FORMAT;
    if (r < 0 || r >= OR_CB_ROWS[ci]) return -OR_ERR_RANGE;
    for (int j = 0; j < OR_CB_WIDTH[ci]; ++j) out[j] = OR_CB[ci][r * OR_CB_WIDTH[ci] + j];
    return OR_CB_WIDTH[ci];
}

int oracle_codebook_rows(const char *name) {
    int ci = or_cb_find(name);
    return ci < 0 ? -OR_ERR_UNKNOWN_FORMAT : OR_CB_ROWS[ci];
}

/* G(name, r): row r of a codebook (NULL when the table is not loaded). */
static const int8_t *G(int ci, uint32_t r) {
    if ((int)r >= OR_CB_ROWS[ci]) return NULL;
    return &OR_CB[ci][r * (uint32_t)OR_CB_WIDTH[ci]];
}

/* S(v): the eight signs 1 - 2*bit(v, j).  SP(v): signs 0..6 from the low
 * seven bits of v and sign 7 from their parity. */
static void S8(uint32_t v, float *s) {
    for (int j = 0; j < 8; ++j) s[j] = 1.0f - 2.0f * (float)field(v, j, 1);
}

static void SP8(uint32_t v, float *s) {
    uint32_t par = 0;
    for (int j = 0; j < 7; ++j) par += field(v, j, 1);
    S8((v & 127u) | ((par % 2u) << 7), s);
}

/* A block is eight groups g of four lanes l; lane i = 4g + l yields outputs
 * 8i .. 8i+7.  For IQ2_XXS, IQ2_XS, IQ2_S, IQ3_XXS and IQ3_S each output is
 * M(M(c, v[j]), s[j]) with the lane's codebook values v, signs s and scale
 * c. */
static void or_lane_signed(float c, const int8_t *v, const float *s, float *y) {
    for (int j = 0; j < 8; ++j) y[j] = M(M(c, (float)v[j]), s[j]);
}

static int dec_iq2_xxs(const uint8_t *b, float *y) {
    float d = H(b);
    for (int g = 0; g < 8; ++g) {
        uint32_t a = U(b + 6 + 8 * g, 4);
        float c = M(M(d, A(0.5f, (float)(a >> 28))), 0.25f);
        for (int l = 0; l < 4; ++l) {
            int i = 4 * g + l;
            const int8_t *v = G(CB_IQ2XXS, b[2 + 8 * g + l]);
            float s[8];
            if (!v) return OR_ERR_UNSUPPORTED_FORMAT;
            SP8(field(a, 7 * l, 7), s);
            or_lane_signed(c, v, s, y + 8 * i);
        }
    }
    return OR_OK;
}

static int dec_iq2_xs(const uint8_t *b, float *y) {
    float d = H(b);
    for (int g = 0; g < 8; ++g)
        for (int l = 0; l < 4; ++l) {
            int i = 4 * g + l;
            uint32_t a = U(b + 2 + 2 * i, 2);
            uint32_t t = field(b[66 + g], 4 * (l / 2), 4);
            float c = M(M(d, A(0.5f, (float)t)), 0.25f);
            const int8_t *v = G(CB_IQ2XS, a % 512u);
            float s[8];
            if (!v) return OR_ERR_UNSUPPORTED_FORMAT;
            SP8(a / 512u, s);
            or_lane_signed(c, v, s, y + 8 * i);
        }
    return OR_OK;
}

static int dec_iq2_s(const uint8_t *b, float *y) {
    float d = H(b);
    for (int g = 0; g < 8; ++g)
        for (int l = 0; l < 4; ++l) {
            int i = 4 * g + l;
            uint32_t r = b[2 + i] + 256u * field(b[66 + g], 2 * l, 2);
            uint32_t t = field(b[74 + g], 4 * (l / 2), 4);
            float c = M(M(d, A(0.5f, (float)t)), 0.25f);
            const int8_t *v = G(CB_IQ2S, r);
            float s[8];
            if (!v) return OR_ERR_UNSUPPORTED_FORMAT;
            S8(b[34 + i], s);
            or_lane_signed(c, v, s, y + 8 * i);
        }
    return OR_OK;
}

static int dec_iq3_xxs(const uint8_t *b, float *y) {
    float d = H(b);
    for (int g = 0; g < 8; ++g) {
        uint32_t a = U(b + 66 + 4 * g, 4);
        float c = M(M(d, A(0.5f, (float)(a >> 28))), 0.5f);
        for (int l = 0; l < 4; ++l) {
            int i = 4 * g + l;
            const int8_t *v0 = G(CB_IQ3XXS, b[2 + 2 * i]), *v1 = G(CB_IQ3XXS, b[3 + 2 * i]);
            int8_t v[8];
            float s[8];
            if (!v0 || !v1) return OR_ERR_UNSUPPORTED_FORMAT;
            for (int j = 0; j < 4; ++j) {
                v[j] = v0[j];
                v[4 + j] = v1[j];
            }
            SP8(field(a, 7 * l, 7), s);
            or_lane_signed(c, v, s, y + 8 * i);
        }
    }
    return OR_OK;
}

static int dec_iq3_s(const uint8_t *b, float *y) {
    float d = H(b);
    for (int g = 0; g < 8; ++g) {
        float c = M(d, (float)(1u + 2u * field(b[106 + g / 2], 4 * (g % 2), 4)));
        for (int l = 0; l < 4; ++l) {
            int i = 4 * g + l;
            int8_t v[8];
            float s[8];
            for (int t = 0; t < 2; ++t) {
                uint32_t r = b[2 + 2 * i + t] + 256u * field(b[66 + g], 2 * l + t, 1);
                const int8_t *row = G(CB_IQ3S, r);
                if (!row) return OR_ERR_UNSUPPORTED_FORMAT;
                for (int j = 0; j < 4; ++j) v[4 * t + j] = row[j];
            }
            S8(b[74 + i], s);
            or_lane_signed(c, v, s, y + 8 * i);
        }
    }
    return OR_OK;
}

/* IQ1_S and IQ1_M: y[8i+j] = M(c, A(v[j], delta)) with v = G(iq1s_grid, r). */
static int or_lane_shifted(float c, uint32_t r, float delta, float *y) {
    const int8_t *v = G(CB_IQ1S, r);
    if (!v) return OR_ERR_UNSUPPORTED_FORMAT;
    for (int j = 0; j < 8; ++j) y[j] = M(c, A((float)v[j], delta));
    return OR_OK;
}

static int dec_iq1_s(const uint8_t *b, float *y) {
    float d = H(b);
    for (int g = 0; g < 8; ++g) {
        uint32_t a = U(b + 34 + 2 * g, 2);
        float c = M(d, (float)(2u * field(a, 12, 3) + 1u));
        float delta = field(a, 15, 1) ? -0.125f : 0.125f;
        for (int l = 0; l < 4; ++l) {
            int i = 4 * g + l;
            uint32_t r = b[2 + i] + 256u * field(a, 3 * l, 3);
            int rc = or_lane_shifted(c, r, delta, y + 8 * i);
            if (rc != OR_OK) return rc;
        }
    }
    return OR_OK;
}

static int dec_iq1_m(const uint8_t *b, float *y) {
    uint32_t w[4], dbits = 0;
    for (int k = 0; k < 4; ++k) {
        w[k] = U(b + 48 + 2 * k, 2);
        dbits += (w[k] >> 12) << (4 * k); /* floor(w[k]/2^12) * 2^(4k) */
    }
    float d = oracle_h2f((uint16_t)dbits);
    for (int g = 0; g < 8; ++g)
        for (int l = 0; l < 4; ++l) {
            int i = 4 * g + l;
            uint32_t a = field(b[32 + i / 2], 4 * (i % 2), 4);
            uint32_t r = b[i] + 256u * (a % 8u);
            uint32_t t = field(w[g / 2], 6 * (g % 2) + 3 * (l / 2), 3);
            float c = M(d, (float)(2u * t + 1u));
            float delta = field(a, 3, 1) ? -0.125f : 0.125f;
            int rc = or_lane_shifted(c, r, delta, y + 8 * i);
            if (rc != OR_OK) return rc;
        }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* The other NInfer grouped schemes and the row-scaled FP8 formats          */
/* ([NINF] sections 4-6.2, 3.4 and the fp8_e4m3fn_row_* description).       */
/* ------------------------------------------------------------------------ */

/* Signed code of a `width`-bit logical word u ([NINF] section 5): u when
 * u < 2^(width-1), else u - 2^width. */
static int32_t or_twos(uint32_t u, int width) {
    return (u < (1u << (width - 1))) ? (int32_t)u : (int32_t)u - (int32_t)(1u << width);
}

/* Logical word k of a packed code plane: bits [width*k, width*k + width) of
 * the little-endian bit stream at `a` (READING: the page gives the words,
 * not their bytes; this is the LSB-first packing of q4_g64_fp16 extended to
 * every width, so fields of 5 and 6 bits may straddle bytes). */
static uint32_t or_stream_word(const uint8_t *a, int k, int width) {
    uint32_t v = 0;
    for (int t = 0; t < width; ++t) {
        int bitpos = width * k + t;
        v |= (uint32_t)field(a[bitpos / 8], bitpos % 8, 1) << t;
    }
    return v;
}

/* q5_g64_fp16 / q6_g64_fp16 / t2_g128_fp16 (READING: a binary16 scale, then
 * the group's codes as a packed plane): w_hat = binary32(s32 * binary32(q))
 * ([NINF] section 6.2) with q the two's-complement code.  t2's word 0b10
 * (-2) is outside the valid artifact language; decoding stays total and
 * gives -2 * s. */
static void dec_grouped_twos(const uint8_t *b, int G, int width, float *y) {
    float s32 = H(b);
    for (int k = 0; k < G; ++k) y[k] = M(s32, (float)or_twos(or_stream_word(b + 2, k, width), width));
}

/* q2_g64_fp16 ([NINF] section 5): the GSQ Q2_0 grid, q = u - 1 for the
 * unsigned 2-bit word u; w_hat = binary32(s32 * binary32(q)). */
static void dec_q2_g64(const uint8_t *b, float *y) {
    float s32 = H(b);
    for (int k = 0; k < 64; ++k) y[k] = M(s32, (float)((int32_t)or_stream_word(b + 2, k, 2) - 1));
}

/* fp8_e4m3fn_row_bf16 / _fp16: one E4M3FN code per element and one row
 * multiplier s32 (already expanded from BF16 or binary16 by the caller):
 * w_hat = binary32(c32 * s32).  A "block" here is one code. */
static void dec_fp8_row(const uint8_t *b, float s32, float *y) { y[0] = M(oracle_e4m3fn(b[0]), s32); }

/* BF16 -> binary32: the 16 bits are the high half of the binary32 pattern
 * ([NINF] section 3.1), exact. */
static float or_bf16_to_f32(uint32_t w) { return or_f32(w << 16); }

static int or_is_fp8_row(const char *name) {
    return strcmp(name, "fp8_e4m3fn_row_bf16") == 0 || strcmp(name, "fp8_e4m3fn_row_fp16") == 0;
}

/* One block of format `name` to binary32.  dw is the nvfp4 divisor, or the
 * expanded row multiplier of an fp8_e4m3fn_row_* code. */
static int or_decode_block(const char *name, const uint8_t *b, float dw, float *y) {
    if (strcmp(name, "gguf:q8_0") == 0 || strcmp(name, "q8_g32_fp16") == 0) dec_q8_0(b, y);
    else if (strcmp(name, "gguf:q4_0") == 0) dec_q4_0(b, y);
    else if (strcmp(name, "gguf:iq4_nl") == 0) dec_iq4_nl(b, y);
    else if (strcmp(name, "gguf:q4_k") == 0) dec_q4_k(b, y);
    else if (strcmp(name, "gguf:q6_k") == 0) dec_q6_k(b, y);
    else if (strcmp(name, "gguf:mxfp4") == 0) dec_mxfp4(b, y);
    else if (strcmp(name, "gguf:nvfp4") == 0) dec_gguf_nvfp4(b, y);
    else if (strcmp(name, "q4_g64_fp16") == 0) dec_q4_g64(b, y);
    else if (strcmp(name, "nvfp4") == 0) dec_nvfp4(b, dw, y);
    else if (strcmp(name, "gguf:q4_1") == 0) dec_q4_1(b, y);
    else if (strcmp(name, "gguf:q5_0") == 0) dec_q5(b, 0, y);
    else if (strcmp(name, "gguf:q5_1") == 0) dec_q5(b, 1, y);
    else if (strcmp(name, "gguf:q8_1") == 0) dec_q8_1(b, y);
    else if (strcmp(name, "gguf:q8_k") == 0) dec_q8_k(b, y);
    else if (strcmp(name, "gguf:q2_k") == 0) dec_q2_k(b, y);
    else if (strcmp(name, "gguf:q3_k") == 0) dec_q3_k(b, y);
    else if (strcmp(name, "gguf:q5_k") == 0) dec_q5_k(b, y);
    else if (strcmp(name, "gguf:iq4_xs") == 0) dec_iq4_xs(b, y);
    else if (strcmp(name, "gguf:tq1_0") == 0) dec_tq1_0(b, y);
    else if (strcmp(name, "gguf:tq2_0") == 0) dec_tq2_0(b, y);
    else if (strcmp(name, "gguf:q1_0") == 0) dec_q1_0(b, y);
    else if (strcmp(name, "gguf:q2_0") == 0) dec_q2_0(b, y);
    else if (strcmp(name, "gguf:iq2_xxs") == 0) return dec_iq2_xxs(b, y);
    else if (strcmp(name, "gguf:iq2_xs") == 0) return dec_iq2_xs(b, y);
    else if (strcmp(name, "gguf:iq2_s") == 0) return dec_iq2_s(b, y);
    else if (strcmp(name, "gguf:iq3_xxs") == 0) return dec_iq3_xxs(b, y);
    else if (strcmp(name, "gguf:iq3_s") == 0) return dec_iq3_s(b, y);
    else if (strcmp(name, "gguf:iq1_s") == 0) return dec_iq1_s(b, y);
    else if (strcmp(name, "gguf:iq1_m") == 0) return dec_iq1_m(b, y);
    else if (strcmp(name, "q2_g64_fp16") == 0) dec_q2_g64(b, y);
    else if (strcmp(name, "q5_g64_fp16") == 0) dec_grouped_twos(b, 64, 5, y);
    else if (strcmp(name, "q6_g64_fp16") == 0) dec_grouped_twos(b, 64, 6, y);
    else if (strcmp(name, "t2_g128_fp16") == 0) dec_grouped_twos(b, 128, 2, y);
    else if (or_is_fp8_row(name)) dec_fp8_row(b, dw, y);
    else return OR_ERR_UNSUPPORTED_FORMAT;
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Top level: validation, block loop, single output cast.                    */
/* ------------------------------------------------------------------------ */

/* Output types: 0 FLOAT, 1 FLOAT16, 2 BFLOAT16, 3 DOUBLE (the four output
 * types of [DQP] "Signature and storage"). */
static int or_out_size(int out_dtype) {
    switch (out_dtype) {
    case 0: return 4;
    case 1: return 2;
    case 2: return 2;
    case 3: return 8;
    default: return 0;
    }
}

static int mul_ovf(uint64_t a, uint64_t b, uint64_t *r) {
    if (a != 0 && b > UINT64_MAX / a) return 1;
    *r = a * b;
    return 0;
}

/* Geometry of a payload under the length rule of [DQP] "Signature and
 * storage": rank >= 1, nonnegative dims, shape[-1] % B == 0 and
 * len(x) == prod(shape[:-1]) * (shape[-1]/B) * S.  For nvfp4 (READING) the
 * payload also carries D >= 1 little-endian FP32 divisors after the blocks;
 * D must divide the row count N = prod(shape[:-1]).  Empty tensors carry no
 * divisor words. */
int oracle_geometry(const char *name, const int64_t *shape, int ndim, uint64_t x_len,
                    uint64_t *nblocks, uint64_t *rows, uint64_t *ndiv) {
    int fi = or_find(name);
    if (fi < 0) return OR_ERR_UNKNOWN_FORMAT;
    if (ndim < 1) return OR_ERR_BAD_RANK;
    if (!shape) return OR_ERR_NULL;
    for (int i = 0; i < ndim; ++i)
        if (shape[i] < 0) return OR_ERR_NEGATIVE_DIM;
    uint64_t B = (uint64_t)OR_FORMATS[fi].B, S = (uint64_t)OR_FORMATS[fi].S;
    uint64_t K = (uint64_t)shape[ndim - 1];
    if (K % B != 0) return OR_ERR_NOT_BLOCK_ALIGNED;
    uint64_t N = 1;
    for (int i = 0; i < ndim - 1; ++i)
        if (mul_ovf(N, (uint64_t)shape[i], &N)) return OR_ERR_OVERFLOW;
    uint64_t nb, bytes, elems;
    if (mul_ovf(N, K / B, &nb)) return OR_ERR_OVERFLOW;
    if (mul_ovf(nb, S, &bytes)) return OR_ERR_OVERFLOW;
    if (mul_ovf(N, K, &elems)) return OR_ERR_OVERFLOW;
    if (bytes > (uint64_t)INT64_MAX || elems > (uint64_t)INT64_MAX / 8) return OR_ERR_OVERFLOW;
    uint64_t D = 0;
    if (strcmp(name, "nvfp4") == 0 && nb > 0) {
        if (x_len < bytes || (x_len - bytes) % 4 != 0) return OR_ERR_LENGTH_MISMATCH;
        D = (x_len - bytes) / 4;
        if (D < 1 || N % D != 0) return OR_ERR_LENGTH_MISMATCH;
    } else if (or_is_fp8_row(name) && nb > 0) {
        /* READING: the N row multipliers follow the code plane */
        if (x_len != bytes + 2u * N) return OR_ERR_LENGTH_MISMATCH;
        D = N;
    } else if (x_len != bytes) {
        return OR_ERR_LENGTH_MISMATCH;
    }
    if (nblocks) *nblocks = nb;
    if (rows) *rows = N;
    if (ndiv) *ndiv = D;
    return OR_OK;
}

static void or_store(int out_dtype, float v, void *y, uint64_t idx) {
    switch (out_dtype) {
    case 0: ((float *)y)[idx] = v; break;
    case 1: ((uint16_t *)y)[idx] = oracle_f32_to_f16(or_bits(v)); break;
    case 2: ((uint16_t *)y)[idx] = oracle_f32_to_bf16(or_bits(v)); break;
    case 3: ((double *)y)[idx] = (double)v; break;
    }
}

/* Decode blocks [b0, b1) of a validated payload into y (which receives
 * (b1-b0)*B values of out_dtype, starting at y[0]).  Blocks are decoded in
 * input order to FLOAT and each value is cast once. */
int oracle_decode_range(const char *name, const int64_t *shape, int ndim, int out_dtype,
                        const uint8_t *x, uint64_t x_len, uint64_t b0, uint64_t b1, void *y) {
    uint64_t nb = 0, N = 0, D = 0;
    int rc = oracle_geometry(name, shape, ndim, x_len, &nb, &N, &D);
    if (rc != OR_OK) return rc;
    if (or_out_size(out_dtype) == 0) return OR_ERR_BAD_DTYPE;
    if (b0 > b1 || b1 > nb) return OR_ERR_RANGE;
    if (b1 == b0) return OR_OK;
    if (!x || !y) return OR_ERR_NULL;
    int fi = or_find(name);
    const or_format *f = &OR_FORMATS[fi];
    if (!f->decoded) return OR_ERR_UNSUPPORTED_FORMAT;
    float blk[256];
    uint64_t bpr = (uint64_t)shape[ndim - 1] / (uint64_t)f->B; /* blocks per row */
    for (uint64_t bi = b0; bi < b1; ++bi) {
        const uint8_t *b = x + bi * (uint64_t)f->S;
        float dw = 1.0f;
        if (strcmp(name, "nvfp4") == 0) {
            /* row r uses divisor floor(r / (N / D)) ([NINF] section 3.3) */
            uint64_t row = bi / bpr;
            uint64_t di = row / (N / D);
            dw = or_f32(U(x + nb * 36u + 4u * di, 4));
        } else if (or_is_fp8_row(name)) {
            /* code bi belongs to row floor(bi / K); its multiplier is word
             * `row` of the plane after the codes */
            uint32_t w = U(x + nb + 2u * (bi / bpr), 2);
            dw = strcmp(name, "fp8_e4m3fn_row_bf16") == 0 ? or_bf16_to_f32(w) : oracle_h2f((uint16_t)w);
        }
        rc = or_decode_block(name, b, dw, blk);
        if (rc != OR_OK) return rc;
        for (int j = 0; j < f->B; ++j)
            or_store(out_dtype, blk[j], y, (bi - b0) * (uint64_t)f->B + (uint64_t)j);
    }
    return OR_OK;
}

/* Whole payload: y receives prod(shape) values of out_dtype. */
int oracle_decode(const char *name, const int64_t *shape, int ndim, int out_dtype,
                  const uint8_t *x, uint64_t x_len, void *y) {
    uint64_t nb = 0;
    int rc = oracle_geometry(name, shape, ndim, x_len, &nb, NULL, NULL);
    if (rc != OR_OK) return rc;
    return oracle_decode_range(name, shape, ndim, out_dtype, x, x_len, 0, nb, y);
}

/* One block to binary32 (before any cast), for pins on hand-built blocks.
 * dw is used by nvfp4 only. */
int oracle_decode_block_f32(const char *name, const uint8_t *b, float dw, float *y) {
    int fi = or_find(name);
    if (fi < 0) return OR_ERR_UNKNOWN_FORMAT;
    if (!b || !y) return OR_ERR_NULL;
    return or_decode_block(name, b, dw, y);
}

/* Kiln group count ([KILN] "Quantization"): ceil(shape[axis]/g) times the
 * product of the other dimensions; the product of no dimensions is 1. */
uint64_t oracle_kiln_group_count(const int64_t *shape, int ndim, int axis, uint64_t g) {
    uint64_t n = ((uint64_t)shape[axis] + g - 1u) / g;
    for (int i = 0; i < ndim; ++i)
        if (i != axis) n *= (uint64_t)shape[i];
    return n;
}

/* ------------------------------------------------------------------------ */
/* grouped_absmax canonical encoder ([NINF] section 7.2), test-only: used to */
/* build q4_g64_fp16 / q8_g32_fp16 payloads for encode/decode round trips.   */
/* ------------------------------------------------------------------------ */

/* round_to_integral_ties_to_even on a binary32 value. */
static float or_rint_even(float x) {
    float a = fabsf(x);
    if (!(a < 8388608.0f)) return x; /* already integral (or non-finite) */
    float fl = floorf(a);
    float frac = a - fl; /* exact for |x| < 2^23 */
    float r;
    if (frac > 0.5f) r = fl + 1.0f;
    else if (frac < 0.5f) r = fl;
    else r = (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
    return (x < 0.0f || (x == 0.0f && signbit(x))) ? -r : r;
}

/* Encode one group of G finite binary32 values with interval [qmin, qmax].
 * Writes the binary16 scale bits and G integer codes. */
int oracle_grouped_absmax_group(const float *x, int G, int qmin, int qmax,
                                uint16_t *scale16_bits, int32_t *codes) {
    float amax = 0.0f;
    for (int i = 0; i < G; ++i) {
        if (!isfinite(x[i])) return OR_ERR_ENCODE;
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        *scale16_bits = 0x0000u;
        for (int i = 0; i < G; ++i) codes[i] = 0;
        return OR_OK;
    }
    float raw_scale32 = amax / (float)qmax;
    uint16_t s16 = oracle_f32_to_f16(or_bits(raw_scale32));
    if ((s16 & 0x7fffu) == 0u) s16 = 0x0001u; /* 2^-24 underflow rescue */
    if ((s16 & 0x7c00u) == 0x7c00u || (s16 & 0x8000u)) return OR_ERR_ENCODE;
    float scale32 = oracle_h2f(s16);
    float inv32 = 1.0f / scale32;
    for (int i = 0; i < G; ++i) {
        float normalized32 = x[i] * inv32;
        float rounded = or_rint_even(normalized32);
        float c = rounded < (float)qmin ? (float)qmin : (rounded > (float)qmax ? (float)qmax : rounded);
        codes[i] = (int32_t)c;
    }
    *scale16_bits = s16;
    return OR_OK;
}

/* Encode a [rows, K] binary32 matrix into a q4_g64_fp16 or q8_g32_fp16
 * payload under this oracle's byte-layout READING.  K must be a multiple of
 * the group size. */
int oracle_encode_grouped(const char *name, const float *x, uint64_t rows, uint64_t K, uint8_t *out) {
    /* qmax of the reference encoder per scheme ([NINF] section 5 table;
     * q8's interval is [-127, 127]) and the code width */
    int width, qmin, qmax;
    uint64_t G = 64u;
    if (!name) return OR_ERR_NULL;
    if (strcmp(name, "q4_g64_fp16") == 0) { width = 4; qmin = -8; qmax = 7; }
    else if (strcmp(name, "q5_g64_fp16") == 0) { width = 5; qmin = -16; qmax = 15; }
    else if (strcmp(name, "q6_g64_fp16") == 0) { width = 6; qmin = -32; qmax = 31; }
    else if (strcmp(name, "q8_g32_fp16") == 0) { width = 8; qmin = -127; qmax = 127; G = 32u; }
    else return OR_ERR_UNSUPPORTED_FORMAT;
    if (K % G != 0) return OR_ERR_NOT_BLOCK_ALIGNED;
    uint64_t S = 2u + G * (uint64_t)width / 8u;
    int32_t codes[64];
    uint64_t nb = rows * (K / G);
    for (uint64_t bi = 0; bi < nb; ++bi) {
        uint16_t s16;
        int rc = oracle_grouped_absmax_group(x + bi * G, (int)G, qmin, qmax, &s16, codes);
        if (rc != OR_OK) return rc;
        uint8_t *b = out + bi * S;
        memset(b, 0, (size_t)S);
        b[0] = (uint8_t)(s16 & 0xffu);
        b[1] = (uint8_t)(s16 >> 8);
        /* codes as width-bit two's-complement words, LSB-first bit stream */
        for (int k = 0; k < (int)G; ++k) {
            uint32_t u = (uint32_t)codes[k] & ((1u << width) - 1u);
            for (int t = 0; t < width; ++t) {
                int bitpos = width * k + t;
                b[2 + bitpos / 8] |= (uint8_t)(((u >> t) & 1u) << (bitpos % 8));
            }
        }
    }
    return OR_OK;
}

/* Array helpers for exhaustive pins. */
void oracle_h2f_array(const uint16_t *in, float *out, uint64_t n) {
    for (uint64_t i = 0; i < n; ++i) out[i] = oracle_h2f(in[i]);
}
void oracle_f32_to_bf16_array(const uint32_t *in, uint16_t *out, uint64_t n) {
    for (uint64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}
void oracle_f32_to_f16_array(const uint32_t *in, uint16_t *out, uint64_t n) {
    for (uint64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Fused consumer reference: the product of activations with decoded         */
/* weights ([NINF] "consuming kernel": a consumer may fuse decode into its   */
/* product, choosing its own staging, reduction order and intermediate       */
/* precision; its result is qualified against an independent oracle).       */
/*                                                                          */
/* READING: the weight operand is DequantizePacked(w, [N, K], T) with T     */
/* FLOAT (the exact binary32 decode) or BFLOAT16 (rounded once to bfloat16, */
/* what a decode-to-bf16 followed by a bf16 product consumes), and the      */
/* activations X are bfloat16 [M, K].  The reference sums the exact products */
/* in binary64:                                                             */
/*     y[m*N + n] = sum_k X[m,k] * W[n,k],   yabs[...] = sum_k |X[m,k] W[n,k]| */
/* (every product of a bfloat16 and a binary32 value is exact in binary64;  */
/* yabs bounds the rounding error of any binary32 evaluation order).        */
/* ------------------------------------------------------------------------ */
static double or_bf16_to_f64(uint16_t h) { return (double)or_f32((uint32_t)h << 16); }

int oracle_matmul_packed(const char *name, uint64_t N, uint64_t K, const uint8_t *w, uint64_t w_len,
                         const uint16_t *x_bf16, uint64_t M, int weight_dtype, double *y, double *yabs) {
    int64_t shape[2] = {(int64_t)N, (int64_t)K};
    uint64_t nb = 0;
    int rc = oracle_geometry(name, shape, 2, w_len, &nb, NULL, NULL);
    if (rc != OR_OK) return rc;
    if (M == 0 || N == 0) return OR_OK;
    if (weight_dtype != 0 && weight_dtype != 2) return OR_ERR_BAD_DTYPE; /* FLOAT or BFLOAT16 */
    if (!x_bf16 || !y || !yabs || (K > 0 && !w)) return OR_ERR_NULL;
    int fi = or_find(name);
    uint64_t bpr = K / (uint64_t)OR_FORMATS[fi].B; /* blocks per weight row */
    float *row = (float *)malloc((size_t)(K ? K : 1) * sizeof(float));
    if (!row) return OR_ERR_NULL;
    for (uint64_t n = 0; n < N; ++n) {
        if (K > 0) {
            rc = oracle_decode_range(name, shape, 2, weight_dtype, w, w_len, n * bpr, (n + 1) * bpr, row);
            if (rc != OR_OK) break;
            if (weight_dtype == 2) /* bfloat16 bit patterns, expanded in place from the top */
                for (uint64_t k = K; k-- > 0;) row[k] = or_f32((uint32_t)((uint16_t *)row)[k] << 16);
        }
        for (uint64_t m = 0; m < M; ++m) {
            double s = 0.0, a = 0.0;
            for (uint64_t k = 0; k < K; ++k) {
                double p = or_bf16_to_f64(x_bf16[m * K + k]) * (double)row[k];
                s += p;
                a += fabs(p);
            }
            y[m * N + n] = s;
            yabs[m * N + n] = a;
        }
    }
    free(row);
    return rc;
}
