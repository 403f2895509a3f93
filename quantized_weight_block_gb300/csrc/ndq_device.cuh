// ndq_device.cuh -- sm_103a decode kernels for packed quantized weights.
//
// Included by one instantiation file per format (ndq_inst_*.cu) so that the
// specialised kernels compile in parallel; everything here has internal
// linkage.
//
// Decode is a streaming, HBM-bound transform (about 2.5 bytes moved per
// element for 4-bit formats to 16-bit outputs, 1-2 FP32 operations per
// element), so the design is about moving bytes, not about tensor cores:
//
//  * persistent CTAs (a grid of SMs x resident CTAs) walk a global list of
//    8192-element tiles that spans one tensor or a whole batch of tensors;
//  * one producer warp per CTA stages each tile's payload bytes (one
//    contiguous span) into shared memory with the Tensor Memory Accelerator
//    (cp.async.bulk, completing on a "full" mbarrier), running up to kStages
//    tiles ahead; it copies the tile's tensor descriptor next to the bytes;
//  * eight consumer warps decode 16-element chunks straight from shared
//    memory (the odd block strides of 17, 18, 34, 36 and 210 bytes are
//    resolved with aligned 32-bit shared loads and funnel shifts), write
//    them with 16-byte vector stores arranged so that each store
//    instruction fills whole 32-byte sectors (adjacent lanes exchange chunk
//    halves, or decode interleaved runs), and release the stage on an
//    "empty" mbarrier.  Consumers never meet at a CTA-wide barrier inside
//    the loop;
//  * nvfp4 to a 16-bit output looks each (scale byte, code) pair up in a
//    per-CTA table of its cast decode; tq1_0 and the FP8 row formats decode
//    16-bit outputs in packed form;
//  * a span that does not start on a 16-byte boundary (an unaligned payload,
//    a ragged last tile) is staged from the 16-byte boundary below it to the
//    one above its end, and decoded at its byte phase within the stage; the
//    extra bytes lie in the same 16-byte lines as payload bytes, hence in
//    mapped memory;
//  * all arithmetic follows the ONNX "DequantizePacked decoding
//    specification" ("Decoding algorithms": every M/A/D rounded separately
//    to binary32, round-to-nearest-even), with explicit __fmul_rn /
//    __fsub_rn / __fdiv_rn and -fmad=false, and a single round-to-nearest-
//    even conversion to the output type.  Integer codes reach FP32 through
//    the exact 2^23 magic-number construction (a byte placed in the low
//    mantissa of 2^23, minus 2^23 plus the code offset), never through a
//    rounding conversion.
//
// Every mbarrier wait is bounded by the global timer; on expiry the warp
// records a fault bit and stops, and the producer waits (bounded) for the
// copies it still has in flight before it exits, so a lost copy cannot hang
// the GPU.

#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ndq_internal.h"

namespace ndq {
namespace {

constexpr int kConsumerWarps = kThreads / 32;     // 8
constexpr uint64_t kWaitLimitNs = 2000000000ull;             // 2 s

// Decode kernel shared memory: decode_stages() payload stages, the header,
// for 16-bit outputs each consumer warp's two output buffers (its 1024
// outputs of a tile, written to global memory by bulk copies), then the
// nvfp4 tables.
constexpr int kWarpOut = kTileElems / kConsumerWarps;               // 1024 outputs per warp per tile
constexpr int kOutBufBytes = kWarpOut * 2;                          // one warp's 16-bit outputs of a tile
constexpr int kOutStageBytes = kConsumerWarps * 2 * kOutBufBytes;  // 32 KB
constexpr int kLutBytes = 256 * 16;                                 // nvfp4 byte table (16 bytes per scale)

static_assert(kInStride >= kMaxTileBytes + 15 + 15 + 12, "stage size");
static_assert(kInStride % 128 == 0, "stage alignment");

// Written by the producer before it arms the stage's full barrier.
struct StageInfo {
    DevTensor t;      // the tile's tensor
    uint64_t block0;  // first block of the tile within the tensor
    uint32_t nb;      // blocks in the tile
    uint32_t phase;   // byte offset of the first block within the stage (0..15)
    uint32_t nv_tab;  // nvfp4: the whole tile uses the divisor the shared table was built for
    uint32_t pad_;
    uint64_t row0;    // fp8 rows: row and column of the tile's first code
    uint64_t col0;
    uint32_t pad[6];
};
static_assert(sizeof(StageInfo) == 128, "StageInfo layout");

struct SmemHdr {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    float lut_iq4[16];  // IQ4_NL table ("Packed layouts and decoding")
    float lut_v[16];    // doubled E2M1 table V ("Ternary and block-floating formats")
    uint32_t tab_bits;  // divisor bits the nvfp4 table was built for
    int32_t tab_valid;
    // nvfp4 per-scale quotients: nv_q[s] = (RN(s/d_w), RN(1.5*s/d_w)); bit s
    // of nv_ok is set when every code of scale byte s is reproduced exactly
    // by nv_q and nv_code (checked against the full table at build time).
    uint32_t nv_ok[8];
    uint2 nv_code[16];  // per E2M1 code: prmt selector of Q1/Q15, bits of +-2^k or +-0
    float2 nv_q[256];
    int32_t pad[6];
    StageInfo info[kStages];
};

constexpr int kHdrBytes = (sizeof(SmemHdr) + 127) / 128 * 128;

__constant__ int8_t c_iq4[16] = {-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113};
__constant__ int8_t c_v[16] = {0, 1, 2, 3, 4, 6, 8, 12, 0, -1, -2, -3, -4, -6, -8, -12};

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, bulk copy, global timer.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: true once the phase with `parity` has completed, false after
// `limit_ns` (by default kWaitLimitNs) of global time.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// TMA bulk copy global -> shared, completing `bytes` of transaction count on
// `bar`.  dst, src and bytes are multiples of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// TMA bulk copy shared -> global of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), tracked in this thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's earlier shared-memory writes before later bulk copies
// (the async proxy) that read them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Shared-memory byte access and exact scalar constructions.
// ---------------------------------------------------------------------------
// 16-bit little-endian field at byte offset `off` of a 16-byte-aligned stage.
// With PH (a stage decoded at a nonzero byte phase) the field may be
// unaligned.
template <bool PH>
__device__ __forceinline__ uint32_t lds_2(const uint8_t* base, uint32_t off) {
    if (PH) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(base + (off & ~3u));
        return __funnelshift_r(w[0], w[1], (off & 3u) * 8u) & 0xffffu;
    }
    return *reinterpret_cast<const uint16_t*>(base + off);
}

// 8 bytes at byte offset `off` of a 16-byte-aligned stage.
__device__ __forceinline__ uint2 lds_8(const uint8_t* base, uint32_t off) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(base + (off & ~3u));
    const uint32_t sh = (off & 3u) * 8u;
    const uint32_t a = w[0], b = w[1], c = w[2];
    return make_uint2(__funnelshift_r(a, b, sh), __funnelshift_r(b, c, sh));
}

// 4 bytes at byte offset `off`.
__device__ __forceinline__ uint32_t lds_4(const uint8_t* base, uint32_t off) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(base + (off & ~3u));
    return __funnelshift_r(w[0], w[1], (off & 3u) * 8u);
}

// prmt.b32 (byte permute of {b, a} by the 4-bit selectors in sel[15:0]; a
// selector's bit 3 replicates the selected byte's top bit).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Two floats to one RNE pair of 16-bit outputs (the first in the low half).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Exact binary16 -> binary32 (the specification's H).
__device__ __forceinline__ float h2f(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// Byte I of w (0..255) as the float 2^23 + byte, minus `bias`: exact for the
// small integers involved (bias = 2^23 + code offset).
template <int I>
__device__ __forceinline__ float byte_minus(uint32_t w, float bias) {
    return __fsub_rn(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | I)), bias);
}

// A signed byte (given as its unsigned byte b) as an exact float.
__device__ __forceinline__ float i8_float(uint32_t b) {
    return __fsub_rn(__uint_as_float(0x4B000000u | (b ^ 0x80u)), 8388736.0f);  // (b ^ 128) - 128
}

// A small unsigned integer u (< 2^23) as an exact float.
__device__ __forceinline__ float small_uint(uint32_t u) {
    return __fsub_rn(__uint_as_float(0x4B000000u | u), 8388608.0f);
}

// Pairs of binary32 values for Blackwell's two-lane FP32 instructions: each
// lane of {sub,mul,fma}.rn.f32x2 is the correctly rounded scalar operation
// (round to nearest even, subnormals kept), so a pair operation gives the
// bits of two __fsub_rn / __fmul_rn / __fmaf_rn at half the issue cost.
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    float2 r;
    asm("{.reg .b64 a, b, r;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "sub.rn.f32x2 r, a, b;\n\t"
        "mov.b64 {%0, %1}, r;}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 r;
    asm("{.reg .b64 a, b, r;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 r, a, b;\n\t"
        "mov.b64 {%0, %1}, r;}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{.reg .b64 a, b, c, r;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "mov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 r, a, b, c;\n\t"
        "mov.b64 {%0, %1}, r;}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

// Bytes I and I+1 of w as the floats 2^23 + byte, minus `bias` (2^23 + code
// offset): exact.
template <int I>
__device__ __forceinline__ float2 bytes_minus2(uint32_t w, float bias) {
    return sub2(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | I)),
                            __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | (I + 1)))),
                make_float2(bias, bias));
}

// Byte I of a and byte I of b, likewise.
template <int I>
__device__ __forceinline__ float2 bytes_minus2(uint32_t a, uint32_t b, float bias) {
    return sub2(make_float2(__uint_as_float(__byte_perm(a, 0x4B000000u, 0x7540u | I)),
                            __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7540u | I))),
                make_float2(bias, bias));
}

// MXFP4 half scale: the FLOAT with bit pattern 0x00200000 * 2^e for e < 2,
// (e-1) * 2^23 otherwise ("Ternary and block-floating formats").
__device__ __forceinline__ float e8m0_half(uint32_t e) {
    return __uint_as_float(e < 2u ? (0x00200000u << e) : ((e - 1u) << 23));
}

// gguf:nvfp4 unsigned-E4M3 half scale: 0 for bytes 0 and 127; otherwise,
// with E = bits 6:3 and m = bits 2:0 (bit 7 ignored), m * 2^-10 when E == 0
// and (1 + m/8) * 2^(E-8) else (exponent field E + 119, mantissa m << 20).
__device__ __forceinline__ float ue4m3_half(uint32_t e) {
    const uint32_t E = (e >> 3) & 15u, m = e & 7u;
    const float r = (E == 0u) ? __fmul_rn(static_cast<float>(m), 0.0009765625f)
                              : __uint_as_float(((E + 119u) << 23) | (m << 20));
    return (e == 0u || e == 127u) ? 0.0f : r;
}

// E4M3FN word (NInfer tensor-formats section 3.3): bias 7, subnormal
// m * 2^-9, e == 15 && m == 7 NaN, sign applies to every word.
__device__ __forceinline__ float e4m3fn(uint32_t w) {
    const uint32_t e = (w >> 3) & 15u, m = w & 7u;
    float mag;
    if (e == 15u && m == 7u)
        mag = __uint_as_float(0x7fc00000u);
    else if (e == 0u)
        mag = __fmul_rn(static_cast<float>(m), 0.001953125f);
    else
        mag = __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (w & 0x80u) ? -mag : mag;
}

// E2M1 word (section 3.3): positive words 0..7 are 0, .5, 1, 1.5, 2, 3, 4, 6;
// bit 3 negates (0x8 is -0).
__device__ __forceinline__ float e2m1(uint32_t c) {
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    const float mag = (e == 0u) ? (m ? 0.5f : 0.0f) : __uint_as_float(((e + 126u) << 23) | (m << 22));
    return (c & 8u) ? -mag : mag;
}

// Little-endian FP32 word at any byte address (global memory).
__device__ __forceinline__ float load_f32_bytes(const uint8_t* p) {
    const uint32_t u = static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) |
                       (static_cast<uint32_t>(p[2]) << 16) | (static_cast<uint32_t>(p[3]) << 24);
    return __uint_as_float(u);
}

// ---------------------------------------------------------------------------
// Per-format chunk decoders: chunk c of a tile = output elements
// CE*c..CE*c+CE-1 of the tile (CE = 16, or 8 for nvfp4: consecutive elements
// of one block), produced from the tile's payload bytes staged at `in` (byte
// phase `ph`: the tile's first block starts at in + ph).  A warp's 32 chunks
// cover 32*CE consecutive outputs; per-chunk work (addresses, scale decode,
// loads) is shared by CE elements.
// ---------------------------------------------------------------------------
struct Ctx {
    const SmemHdr* H;
    const float* tab;  // nvfp4 quotient table, or nullptr for per-element division
    const uint8_t* divs;
    uint64_t block0;
    uint64_t blocks_per_div;
    const IqGrids* grids;  // IQ codebooks
    uint64_t n_el;         // fp8 rows: codes in the tensor (the last 16-code unit may be partial)
    uint64_t row0;         // fp8 rows: row and column of the code at block0
    uint64_t col0;
};

__host__ __device__ constexpr bool is_fp8_row(int f) { return f == KF_FP8_ROW_BF16 || f == KF_FP8_ROW_FP16; }

// Codes of an fp8 row tensor: its row multipliers start right after the code
// plane.  0 for every other format.
__device__ __forceinline__ uint64_t code_count(const DevTensor& t) {
    return is_fp8_row(t.fmt) ? static_cast<uint64_t>(reinterpret_cast<uintptr_t>(t.divs) -
                                                      reinterpret_cast<uintptr_t>(t.x))
                             : 0u;
}

// 16 bytes at byte offset `off` of a 16-byte-aligned stage (ALIGNED: off is a
// multiple of 16, one 16-byte load).
template <bool ALIGNED>
__device__ __forceinline__ uint4 lds_16(const uint8_t* base, uint32_t off) {
    if (ALIGNED) return *reinterpret_cast<const uint4*>(base + off);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(base + (off & ~3u));
    const uint32_t sh = (off & 3u) * 8u;
    const uint32_t a = w[0], b = w[1], c = w[2], d = w[3], e = w[4];
    return make_uint4(__funnelshift_r(a, b, sh), __funnelshift_r(b, c, sh), __funnelshift_r(c, d, sh),
                      __funnelshift_r(d, e, sh));
}

// Four bytes of w (values < 256) as exact floats minus the code offset, times
// d: v[i] = M(d, byte_i - offset) with bias = 2^23 + offset.
__device__ __forceinline__ void mul4(float d, uint32_t w, float bias, float* v) {
    const float2 dd = make_float2(d, d);
    const float2 a = mul2(dd, bytes_minus2<0>(w, bias)), b = mul2(dd, bytes_minus2<2>(w, bias));
    v[0] = a.x;
    v[1] = a.y;
    v[2] = b.x;
    v[3] = b.y;
}

// v[i] = fma(a, byte_i - offset, c): one rounding of a * byte + c, used only
// where the product is exact in binary32.
__device__ __forceinline__ void fma4(float a, uint32_t w, float bias, float c, float* v) {
    const float2 aa = make_float2(a, a), cc = make_float2(c, c);
    const float2 x = fma2(aa, bytes_minus2<0>(w, bias), cc), y = fma2(aa, bytes_minus2<2>(w, bias), cc);
    v[0] = x.x;
    v[1] = x.y;
    v[2] = y.x;
    v[3] = y.y;
}

// Table lookup of four nibbles (bytes of w) scaled by d: v[i] = M(d, T[n_i]).
__device__ __forceinline__ void lut4(const float* T, float d, uint32_t w, float* v) {
    const float2 dd = make_float2(d, d);
    const float2 a = mul2(dd, make_float2(T[w & 15u], T[(w >> 8) & 15u]));
    const float2 b = mul2(dd, make_float2(T[(w >> 16) & 15u], T[(w >> 24) & 15u]));
    v[0] = a.x;
    v[1] = a.y;
    v[2] = b.x;
    v[3] = b.y;
}

template <int F>
struct Fmt;

// gguf:q8_0 / q8_g32_fp16: y[j] = M(d, q[j]), q signed bytes; chunk c&1 holds
// q[16*(c&1) .. +16].
template <>
struct Fmt<KF_Q8_0> {
    static constexpr int B = 32, S = 34, CE = 16, CPB = 2;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 1) * S;
        const float d = h2f(lds_2<PH>(in, off));
        const uint4 q = lds_16<false>(in, off + 2u + 16u * (c & 1u));
        const float bias = 8388736.0f;  // 2^23 + 128; XOR 0x80 maps signed to offset-128
        mul4(d, q.x ^ 0x80808080u, bias, v);
        mul4(d, q.y ^ 0x80808080u, bias, v + 4);
        mul4(d, q.z ^ 0x80808080u, bias, v + 8);
        mul4(d, q.w ^ 0x80808080u, bias, v + 12);
    }
};

// Nibble plane p (0 = low, 1 = high) of 16 consecutive code bytes, as bytes.
__device__ __forceinline__ uint4 nib_plane16(uint4 q, uint32_t p) {
    const uint32_t s = 4u * p;
    return make_uint4((q.x >> s) & 0x0F0F0F0Fu, (q.y >> s) & 0x0F0F0F0Fu, (q.z >> s) & 0x0F0F0F0Fu,
                      (q.w >> s) & 0x0F0F0F0Fu);
}

// gguf:q4_0: v = P(q,4,16) (16 low nibbles, then 16 high nibbles), so chunk
// c&1 is plane c&1 of the 16 code bytes; y[j] = M(d, v[j] - 8).
template <>
struct Fmt<KF_Q4_0> {
    static constexpr int B = 32, S = 18, CE = 16, CPB = 2;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 1) * S;
        const float d = h2f(lds_2<PH>(in, off));
        const uint4 n = nib_plane16(lds_16<false>(in, off + 2u), c & 1u);
        const float bias = 8388616.0f;  // 2^23 + 8
        mul4(d, n.x, bias, v);
        mul4(d, n.y, bias, v + 4);
        mul4(d, n.z, bias, v + 8);
        mul4(d, n.w, bias, v + 12);
    }
};

// gguf:iq4_nl: v = P(q,4,16); y[j] = M(d, IQ4[v[j]]).
template <>
struct Fmt<KF_IQ4_NL> {
    static constexpr int B = 32, S = 18, CE = 16, CPB = 2;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 1) * S;
        const float d = h2f(lds_2<PH>(in, off));
        const uint4 n = nib_plane16(lds_16<false>(in, off + 2u), c & 1u);
        const float* T = x.H->lut_iq4;
        lut4(T, d, n.x, v);
        lut4(T, d, n.y, v + 4);
        lut4(T, d, n.z, v + 8);
        lut4(T, d, n.w, v + 12);
    }
};

// gguf:mxfp4: d = E8M0 half scale; v = P(q,4,16); y[j] = M(d, V[v[j]]).
template <>
struct Fmt<KF_MXFP4> {
    static constexpr int B = 32, S = 17, CE = 16, CPB = 2;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 1) * S;
        const float d = e8m0_half(in[off]);
        const uint4 n = nib_plane16(lds_16<false>(in, off + 1u), c & 1u);
        const float* T = x.H->lut_v;
        lut4(T, d, n.x, v);
        lut4(T, d, n.y, v + 4);
        lut4(T, d, n.z, v + 8);
        lut4(T, d, n.w, v + 12);
    }
};

// gguf:nvfp4: chunk c&3 is group g of 16 values: d = unsigned-E4M3 half scale
// of scales[g]; v = P(q[8g:8g+8],4,8) (8 low nibbles, then 8 high);
// y[16g+j] = M(d, V[v[j]]).
template <>
struct Fmt<KF_GGUF_NVFP4> {
    static constexpr int B = 64, S = 36, CE = 16, CPB = 4;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 2) * S, g = c & 3u;
        const float d = ue4m3_half(in[off + g]);
        const uint2 q = lds_8(in, off + 4u + 8u * g);
        const float* T = x.H->lut_v;
        lut4(T, d, q.x & 0x0F0F0F0Fu, v);
        lut4(T, d, q.y & 0x0F0F0F0Fu, v + 4);
        lut4(T, d, (q.x >> 4) & 0x0F0F0F0Fu, v + 8);
        lut4(T, d, (q.y >> 4) & 0x0F0F0F0Fu, v + 12);
    }
};

// nvfp4 (NInfer section 3.3): W = e2m1(c) * e4m3fn(s) / d_w, the product exact
// and the quotient rounded once.  Chunk c&3 is group g (scale byte g, codes
// laid out as gguf:nvfp4).  With the per-scale quotients (the tile uses the
// divisor the shared tables were built for, and scale byte s passed the
// build-time check), the element is Q_m(s) * (+-2^k or +-0) for the code's
// E2M1 magnitude 2^k * m; failing that, the full quotient table
// tab[16*s + c]; for a tile that spans two divisors, a division.
template <>
struct Fmt<KF_NVFP4> {
    // 8-element chunks: this decoder needs more registers than the others,
    // and at 16 elements per chunk it loses a resident CTA per SM.
    static constexpr int B = 64, S = 36, CE = 8, CPB = 8;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        // chunk c&7: group g = (c&7)>>1 (scale byte g), plane (c&1) of its 8 code bytes
        const uint32_t off = ph + (c >> 3) * S, cc = c & 7u, g = cc >> 1;
        const uint32_t s = in[off + g];
        const uint2 q = lds_8(in, off + 4u + 8u * g);
        const uint32_t sh = 4u * (cc & 1u);
        const uint32_t a = (q.x >> sh) & 0x0F0F0F0Fu, b = (q.y >> sh) & 0x0F0F0F0Fu;
        if (x.tab && ((x.H->nv_ok[s >> 5] >> (s & 31u)) & 1u)) {
            // Every E2M1 magnitude is 2^k * m, m in {1, 1.5}: the element is the
            // exact quotient Q_m(s) times +-2^k (or +-0); both lookups are
            // 16-entry tables, so a warp's accesses never conflict in banks.
            const float2 qq = x.H->nv_q[s];
            const uint32_t q1 = __float_as_uint(qq.x), q15 = __float_as_uint(qq.y);
            const uint2* K = x.H->nv_code;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint2 ka = K[(a >> (8 * i)) & 15u], kb = K[(b >> (8 * i)) & 15u];
                v[i] = __fmul_rn(__uint_as_float(__byte_perm(q1, q15, ka.x)), __uint_as_float(ka.y));
                v[4 + i] = __fmul_rn(__uint_as_float(__byte_perm(q1, q15, kb.x)), __uint_as_float(kb.y));
            }
        } else if (x.tab) {
            const float* T = x.tab + s * 16u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[i] = T[(a >> (8 * i)) & 15u];
                v[4 + i] = T[(b >> (8 * i)) & 15u];
            }
        } else {  // divisor of this block, then divide
            const float dw = load_f32_bytes(x.divs + 4u * ((x.block0 + (c >> 3)) / x.blocks_per_div));
            const float sc = e4m3fn(s);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[i] = __fdiv_rn(__fmul_rn(e2m1((a >> (8 * i)) & 15u), sc), dw);
                v[4 + i] = __fdiv_rn(__fmul_rn(e2m1((b >> (8 * i)) & 15u), sc), dw);
            }
        }
    }
};

// gguf:q4_k: v = P(q,4,32); 6-bit a[k], m[k] from the 12 scale bytes;
// y[j] = D(M(M(d, a[k]), v[j]), M(dmin, m[k])), k = floor(j/32).
// Chunk c&15 = elements 16cc..16cc+15: sub-block k = cc>>1, byte group cc>>2
// (32 bytes), plane (cc>>1)&1, bytes 16*(cc&1) of the group.
template <>
struct Fmt<KF_Q4_K> {
    static constexpr int B = 256, S = 144, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, k = cc >> 1;
        // Block header: d, dmin and the scale bytes s[0..11] as three words
        // (byte j of word w is s[4w + j]); one 16-byte load when aligned.
        const uint4 hdr = lds_16<!PH>(in, off);
        const float d = h2f(hdr.x & 0xffffu), dmin = h2f(hdr.x >> 16);
        // With j = k mod 4, byte j of each word is s[j], s[j+4], s[j+8].  Both
        // unpack rules are formed and one is selected, so the lanes of a warp
        // (k = (lane mod 16)/2) do not diverge.
        const uint32_t j8 = 8u * (k & 3u);
        const uint32_t b0 = (hdr.y >> j8) & 0xffu, b1 = (hdr.z >> j8) & 0xffu, b2 = (hdr.w >> j8) & 0xffu;
        const bool lo = k < 4u;
        const uint32_t sa = lo ? (b0 & 63u) : ((b2 & 15u) | ((b0 >> 6) << 4));
        const uint32_t sm = lo ? (b1 & 63u) : ((b2 >> 4) | ((b1 >> 6) << 4));
        const float da = __fmul_rn(d, small_uint(sa));
        const float ndm = -__fmul_rn(dmin, small_uint(sm));
        const uint4 n = nib_plane16(lds_16<!PH>(in, off + 16u + 32u * (cc >> 2) + 16u * (cc & 1u)), k & 1u);
        // D(M(da, v), dm) as one fused multiply-add: da = M(d, a) has at most
        // 17 significant bits and v at most 4, so M(da, v) is exact in
        // binary32 and the FMA rounds the same exact difference once (the
        // product cannot overflow, and inf/NaN/zero cases match term by term).
        const float bias = 8388608.0f;  // 2^23
        fma4(da, n.x, bias, ndm, v);
        fma4(da, n.y, bias, ndm, v + 4);
        fma4(da, n.z, bias, ndm, v + 8);
        fma4(da, n.w, bias, ndm, v + 12);
    }
};

// gguf:q6_k: l = P(low,4,64), h = P(high,2,32), s = scales[floor(j/16)] signed;
// y[j] = M(M(d, s), l[j] + 16 h[j] - 32).  Chunk c&15 = elements
// 16cc..16cc+15 shares scale cc: low bytes 64*(cc>>3) + 16*(cc&3), plane
// (cc>>2)&1; high bytes 32*(cc>>3) + 16*(cc&1), 2-bit plane (cc>>1)&3.
template <>
struct Fmt<KF_Q6_K> {
    static constexpr int B = 256, S = 210, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, gi = cc >> 3;
        const float d = h2f(lds_2<PH>(in, off + 208u));
        const float ds = __fmul_rn(d, i8_float(in[off + 192u + cc]));
        const uint4 lo = lds_16<false>(in, off + 64u * gi + 16u * (cc & 3u));
        const uint4 hi = lds_16<false>(in, off + 128u + 32u * gi + 16u * (cc & 1u));
        const uint32_t pl = 4u * ((cc >> 2) & 1u), phh = 2u * ((cc >> 1) & 3u);
        const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w}, hw[4] = {hi.x, hi.y, hi.z, hi.w};
        const float bias = 8388640.0f;  // 2^23 + 32
#pragma unroll
        for (int q = 0; q < 4; ++q)
            mul4(ds, ((lw[q] >> pl) & 0x0F0F0F0Fu) | (((hw[q] >> phh) & 0x03030303u) << 4), bias, v + 4 * q);
    }
    // The two runs of lane h = c & 1 within the pair of chunks c & ~1, c | 1
    // (scales cc & ~1 and cc | 1; their low and high bytes are 32 consecutive
    // bytes each): v[0..7] = pair elements 8h..8h+7 (first scale), v[8..15]
    // = elements 24-8h..31-8h (second scale).
    template <bool PH>
    __device__ __forceinline__ static void pair_runs(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                     const Ctx&) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 14u, gi = cc >> 3, h = c & 1u;
        const float d = h2f(lds_2<PH>(in, off + 208u));
        const float ds0 = __fmul_rn(d, i8_float(in[off + 192u + cc]));
        const float ds1 = __fmul_rn(d, i8_float(in[off + 193u + cc]));
        const uint32_t lb = off + 64u * gi + 16u * (cc & 3u), hb = off + 128u + 32u * gi;
        const uint2 la = lds_8(in, lb + 8u * h), lbb = lds_8(in, lb + 24u - 8u * h);
        const uint2 ha = lds_8(in, hb + 8u * h), hbb = lds_8(in, hb + 24u - 8u * h);
        const uint32_t pl = 4u * ((cc >> 2) & 1u), phh = 2u * ((cc >> 1) & 3u);
        const uint32_t lw[4] = {la.x, la.y, lbb.x, lbb.y}, hw[4] = {ha.x, ha.y, hbb.x, hbb.y};
        const float bias = 8388640.0f;  // 2^23 + 32
#pragma unroll
        for (int q = 0; q < 4; ++q)
            mul4(q < 2 ? ds0 : ds1, ((lw[q] >> pl) & 0x0F0F0F0Fu) | (((hw[q] >> phh) & 0x03030303u) << 4), bias,
                 v + 4 * q);
    }
};

// q4_g64_fp16 (NInfer sections 5-6.2): w = binary32(s32 * q), q the 4-bit
// two's-complement code; element k sits in bits 4*(k mod 2) of code byte
// floor(k/2) (layout reading), so chunk c&3 is code bytes 8*(c&3)..+8.
// XOR 8 maps two's complement to offset-8.
template <>
struct Fmt<KF_Q4_G64> {
    static constexpr int B = 64, S = 34, CE = 16, CPB = 4;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 2) * S;
        const float s = h2f(lds_2<PH>(in, off));
        const uint2 q = lds_8(in, off + 2u + 8u * (c & 3u));
        const float bias = 8388616.0f;  // 2^23 + 8
        const uint32_t wv[2] = {q.x, q.y};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t lo = (wv[h] & 0x0F0F0F0Fu) ^ 0x08080808u, hi = ((wv[h] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
            float* o = v + 8 * h;
            const float2 ss = make_float2(s, s);
            const float2 a = mul2(ss, bytes_minus2<0>(lo, hi, bias)), b = mul2(ss, bytes_minus2<1>(lo, hi, bias));
            const float2 e = mul2(ss, bytes_minus2<2>(lo, hi, bias)), f = mul2(ss, bytes_minus2<3>(lo, hi, bias));
            o[0] = a.x;
            o[1] = a.y;
            o[2] = b.x;
            o[3] = b.y;
            o[4] = e.x;
            o[5] = e.y;
            o[6] = f.x;
            o[7] = f.y;
        }
    }
};

// ---------------------------------------------------------------------------
// The other simple gguf profiles ("Mathematical decoding rules").  Where a
// rule adds or subtracts after an exact product (an fp16 scale times an
// integer of at most 5 bits, or a 17-bit sub-scale product times at most 5
// bits), the product and the sum are formed by one FMA: the product is exact
// in binary32, so the single rounding is the rule's.
// ---------------------------------------------------------------------------

// 4 bits of `b` (bits 0..3) spread to bit 4 of each byte: the 5th code bit.
__device__ __forceinline__ uint32_t spread4_b4(uint32_t b) { return ((b * 0x00204081u) & 0x01010101u) << 4; }

// gguf:q4_1: v = P(q,4,16); y[j] = A(M(d, v[j]), m).
template <>
struct Fmt<KF_Q4_1> {
    static constexpr int B = 32, S = 20, CE = 16, CPB = 2;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 1) * S;
        const float d = h2f(lds_2<PH>(in, off)), m = h2f(lds_2<PH>(in, off + 2u));
        const uint4 n = nib_plane16(lds_16<false>(in, off + 4u), c & 1u);
        const float bias = 8388608.0f;  // 2^23
        fma4(d, n.x, bias, m, v);
        fma4(d, n.y, bias, m, v + 4);
        fma4(d, n.z, bias, m, v + 8);
        fma4(d, n.w, bias, m, v + 12);
    }
};

// gguf:q5_0 / q5_1: v = P(q,4,16) + 16*bit(U(high), j); Q5_0 y = M(d, v-16),
// Q5_1 y = A(M(d, v), m).  Chunk c&1 = plane c&1, high bits 16*(c&1)...
template <bool AFF>
struct Q5Impl {
    static constexpr int S = AFF ? 24 : 22;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v) {
        const uint32_t off = ph + (c >> 1) * S, o = AFF ? 4u : 2u;
        const float d = h2f(lds_2<PH>(in, off));
        const float m = AFF ? h2f(lds_2<PH>(in, off + 2u)) : 0.0f;
        const uint32_t hb = lds_4(in, off + o) >> (16u * (c & 1u));
        const uint4 n = nib_plane16(lds_16<false>(in, off + o + 4u), c & 1u);
        const uint32_t w[4] = {n.x, n.y, n.z, n.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t u = w[q] | spread4_b4((hb >> (4 * q)) & 15u);
            if (AFF) {
                fma4(d, u, 8388608.0f, m, v + 4 * q);  // 2^23
            } else {
                mul4(d, u, 8388624.0f, v + 4 * q);  // 2^23 + 16
            }
        }
    }
};
template <>
struct Fmt<KF_Q5_0> {
    static constexpr int B = 32, S = 22, CE = 16, CPB = 2;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        Q5Impl<false>::chunk<PH>(in, ph, c, v);
    }
};
template <>
struct Fmt<KF_Q5_1> {
    static constexpr int B = 32, S = 24, CE = 16, CPB = 2;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        Q5Impl<true>::chunk<PH>(in, ph, c, v);
    }
};

// gguf:q8_1 (h d, s; i8 q[32]) and gguf:q8_k (f d; i8 q[256]; i16 sums[16]):
// y[j] = M(d, q[j]); the cached sum fields are never read.
template <>
struct Fmt<KF_Q8_1> {
    static constexpr int B = 32, S = 36, CE = 16, CPB = 2;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 1) * S;
        const float d = h2f(lds_2<PH>(in, off));
        const uint4 q = lds_16<false>(in, off + 4u + 16u * (c & 1u));
        const float bias = 8388736.0f;  // 2^23 + 128
        mul4(d, q.x ^ 0x80808080u, bias, v);
        mul4(d, q.y ^ 0x80808080u, bias, v + 4);
        mul4(d, q.z ^ 0x80808080u, bias, v + 8);
        mul4(d, q.w ^ 0x80808080u, bias, v + 12);
    }
};
template <>
struct Fmt<KF_Q8_K> {
    static constexpr int B = 256, S = 292, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 4) * S;
        const float d = __uint_as_float(lds_4(in, off));
        const uint4 q = lds_16<false>(in, off + 4u + 16u * (c & 15u));
        const float bias = 8388736.0f;
        mul4(d, q.x ^ 0x80808080u, bias, v);
        mul4(d, q.y ^ 0x80808080u, bias, v + 4);
        mul4(d, q.z ^ 0x80808080u, bias, v + 8);
        mul4(d, q.w ^ 0x80808080u, bias, v + 12);
    }
};

// 2-bit plane p of 16 code bytes, as bytes (P(q,2,32) layout).
__device__ __forceinline__ uint4 plane2_16(uint4 q, uint32_t p) {
    const uint32_t s = 2u * p;
    return make_uint4((q.x >> s) & 0x03030303u, (q.y >> s) & 0x03030303u, (q.z >> s) & 0x03030303u,
                      (q.w >> s) & 0x03030303u);
}

// Bit b of 16 mask bytes, as bytes (P(mask,1,32) layout).
__device__ __forceinline__ uint4 plane1_16(uint4 q, uint32_t b) {
    return make_uint4((q.x >> b) & 0x01010101u, (q.y >> b) & 0x01010101u, (q.z >> b) & 0x01010101u,
                      (q.w >> b) & 0x01010101u);
}

// gguf:q2_k: v = P(q,2,32), s = scales[floor(j/16)];
// y[j] = D(M(M(d, s mod 16), v[j]), M(dmin, floor(s/16))).  Chunk cc = scale
// cc; code bytes 32*(cc>>3) + 16*(cc&1), plane (cc>>1)&3.
template <>
struct Fmt<KF_Q2_K> {
    static constexpr int B = 256, S = 84, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u;
        const uint32_t sc = in[off + cc];
        const float d = h2f(lds_2<PH>(in, off + 80u)), dmin = h2f(lds_2<PH>(in, off + 82u));
        const float ds = __fmul_rn(d, small_uint(sc & 15u));
        const float ndm = -__fmul_rn(dmin, small_uint(sc >> 4));
        const uint4 n = plane2_16(lds_16<false>(in, off + 16u + 32u * (cc >> 3) + 16u * (cc & 1u)), (cc >> 1) & 3u);
        const float bias = 8388608.0f;
        fma4(ds, n.x, bias, ndm, v);
        fma4(ds, n.y, bias, ndm, v + 4);
        fma4(ds, n.z, bias, ndm, v + 8);
        fma4(ds, n.w, bias, ndm, v + 12);
    }
};

// gguf:q3_k: v = P(q,2,32), h = P(mask,1,32), l = P(b[96:104],4,8),
// a = P(b[104:108],2,4); s = l[k] + 16 a[k] - 32 with k = floor(j/16);
// y[j] = M(M(d, s), v[j] - 4*(1 - h[j])).  Chunk cc: scale k = cc; codes as
// q2_k at byte 32; mask bit cc>>1 of mask bytes 16*(cc&1)...
template <>
struct Fmt<KF_Q3_K> {
    static constexpr int B = 256, S = 110, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u;
        const float d = h2f(lds_2<PH>(in, off + 108u));
        const uint32_t l = (in[off + 96u + (cc & 7u)] >> (4u * (cc >> 3))) & 15u;
        const uint32_t a = (in[off + 104u + (cc & 3u)] >> (2u * (cc >> 2))) & 3u;
        const float ds = __fmul_rn(d, __fsub_rn(__uint_as_float(0x4B000000u | (l + 16u * a)), 8388640.0f));  // - 32
        const uint4 vq = plane2_16(lds_16<false>(in, off + 32u + 32u * (cc >> 3) + 16u * (cc & 1u)), (cc >> 1) & 3u);
        const uint4 hm = plane1_16(lds_16<false>(in, off + 16u * (cc & 1u)), cc >> 1);
        // v - 4*(1 - h) = (v + 4h) - 4
        mul4(ds, vq.x | (hm.x << 2), 8388612.0f, v);  // 2^23 + 4
        mul4(ds, vq.y | (hm.y << 2), 8388612.0f, v + 4);
        mul4(ds, vq.z | (hm.z << 2), 8388612.0f, v + 8);
        mul4(ds, vq.w | (hm.w << 2), 8388612.0f, v + 12);
    }
};

// gguf:q5_k: v = P(q,4,32) + 16*P(high,1,32); a, m as q4_k;
// y[j] = D(M(M(d, a[k]), v[j]), M(dmin, m[k])).  Chunk cc: sub-block k = cc>>1,
// codes 48 + 32*(cc>>2) + 16*(cc&1) plane k&1, high bit k of bytes 16 + 16*(cc&1).
template <>
struct Fmt<KF_Q5_K> {
    static constexpr int B = 256, S = 176, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, k = cc >> 1;
        const uint4 hdr = lds_16<!PH>(in, off);
        const float d = h2f(hdr.x & 0xffffu), dmin = h2f(hdr.x >> 16);
        const uint32_t j8 = 8u * (k & 3u);
        const uint32_t b0 = (hdr.y >> j8) & 0xffu, b1 = (hdr.z >> j8) & 0xffu, b2 = (hdr.w >> j8) & 0xffu;
        const bool lo = k < 4u;
        const uint32_t sa = lo ? (b0 & 63u) : ((b2 & 15u) | ((b0 >> 6) << 4));
        const uint32_t sm = lo ? (b1 & 63u) : ((b2 >> 4) | ((b1 >> 6) << 4));
        const float da = __fmul_rn(d, small_uint(sa));
        const float ndm = -__fmul_rn(dmin, small_uint(sm));
        const uint4 n = nib_plane16(lds_16<!PH>(in, off + 48u + 32u * (cc >> 2) + 16u * (cc & 1u)), k & 1u);
        const uint4 hb = plane1_16(lds_16<!PH>(in, off + 16u + 16u * (cc & 1u)), k);
        const float bias = 8388608.0f;
        fma4(da, n.x | (hb.x << 4), bias, ndm, v);
        fma4(da, n.y | (hb.y << 4), bias, ndm, v + 4);
        fma4(da, n.z | (hb.z << 4), bias, ndm, v + 8);
        fma4(da, n.w | (hb.w << 4), bias, ndm, v + 12);
    }
};

// gguf:iq4_xs: v = P(q,4,16); s[k] = field(scales[k/2], 4(k mod 2), 4)
// + 16*field(high, 2k, 2) - 32; y[j] = M(M(d, s[floor(j/32)]), IQ4[v[j]]).
// Chunk cc: k = cc>>1, plane cc&1 of code bytes 16k...
template <>
struct Fmt<KF_IQ4_XS> {
    static constexpr int B = 256, S = 136, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, k = cc >> 1;
        const float d = h2f(lds_2<PH>(in, off));
        const uint32_t high = lds_2<PH>(in, off + 2u);
        const uint32_t lo4 = (in[off + 4u + (k >> 1)] >> (4u * (k & 1u))) & 15u;
        const uint32_t sc = lo4 | (((high >> (2u * k)) & 3u) << 4);  // s + 32
        const float ds = __fmul_rn(d, __fsub_rn(__uint_as_float(0x4B000000u | sc), 8388640.0f));
        const uint4 n = nib_plane16(lds_16<false>(in, off + 8u + 16u * k), cc & 1u);
        const float* T = x.H->lut_iq4;
        lut4(T, ds, n.x, v);
        lut4(T, ds, n.y, v + 4);
        lut4(T, ds, n.z, v + 8);
        lut4(T, ds, n.w, v + 12);
    }
};

// gguf:tq1_0: outputs in three sequences (start, width, count) = (0,32,5),
// (32,16,5), (48,4,4), plane p before lane j: M(d, floor(3*((b*3^p) mod 256)
// /256) - 1).  Chunks 0..9: p = cc>>1, bytes 16*(cc&1)...; 10..14: p = cc-10,
// bytes 32..47; 15: element i has p = i/4 and byte 48 + i%4.
template <>
struct Fmt<KF_TQ1_0> {
    static constexpr int B = 256, S = 54, CE = 16, CPB = 16;
    __device__ __forceinline__ static float trit(uint32_t byte, uint32_t pw) {
        const uint32_t t = ((((byte * pw) & 255u) * 3u) >> 8);  // 0, 1 or 2
        return __fsub_rn(__uint_as_float(0x4B000000u | t), 8388609.0f);  // t - 1, exact
    }
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u;
        const float d = h2f(lds_2<PH>(in, off + 52u));
        const uint32_t start = cc < 10u ? 16u * (cc & 1u) : (cc < 15u ? 32u : 48u);
        const uint4 q = lds_16<false>(in, off + start);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        if (cc < 15u) {
            const uint32_t p = cc < 10u ? (cc >> 1) : (cc - 10u);
            const uint32_t pw = p == 0u ? 1u : p == 1u ? 3u : p == 2u ? 9u : p == 3u ? 27u : 81u;
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(d, trit((w[i >> 2] >> (8 * (i & 3))) & 255u, pw));
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t pw = (i >> 2) == 0 ? 1u : (i >> 2) == 1 ? 3u : (i >> 2) == 2 ? 9u : 27u;
                v[i] = __fmul_rn(d, trit((w[0] >> (8 * (i & 3))) & 255u, pw));
            }
        }
    }
    // The same chunk as 16-bit outputs of type O (pairs in w[0..7]).  A
    // block has three outputs, cast(M(d, -1)), cast(M(d, +0)) and
    // cast(M(d, 1)), held as a 6-byte table; each group of 4 codes (4 bytes
    // sharing one power 3^p) gets its trits two at a time in 16-bit lanes,
    // ((b * 3^p) mod 256) * 3 >> 8 (b * 81 < 2^16, so lanes do not carry),
    // and one prmt per output pair looks up the table.
    template <bool PH, int O>
    __device__ __forceinline__ static void chunk16(const uint8_t* in, uint32_t ph, uint32_t c, uint32_t* w,
                                                   const Ctx&) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u;
        const float d = h2f(lds_2<PH>(in, off + 52u));
        const uint32_t start = cc < 10u ? 16u * (cc & 1u) : (cc < 15u ? 32u : 48u);
        const uint4 q = lds_16<false>(in, off + start);
        const uint32_t p = cc < 10u ? (cc >> 1) : (cc - 10u);
        const uint32_t pw = p == 0u ? 1u : p == 1u ? 3u : p == 2u ? 9u : p == 3u ? 27u : 81u;
        const float dm = __fmul_rn(d, -1.0f), d0 = __fmul_rn(d, 0.0f), d1 = __fmul_rn(d, 1.0f);
        const uint32_t ta = (O == KO_BF16) ? pack_bf16(dm, d0) : pack_f16(dm, d0);
        const uint32_t tb = (O == KO_BF16) ? pack_bf16(d1, 0.0f) : pack_f16(d1, 0.0f);
        const bool last = cc == 15u;  // element i: byte 48 + i%4, power 3^(i/4)
        const uint32_t g[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t W = last ? q.x : g[k];
            const uint32_t P = last ? (k == 0 ? 1u : k == 1 ? 3u : k == 2 ? 9u : 27u) : pw;
            const uint32_t lo = ((W & 0x00FF00FFu) * P) & 0x00FF00FFu;         // bytes 0, 2
            const uint32_t hi = (((W >> 8) & 0x00FF00FFu) * P) & 0x00FF00FFu;  // bytes 1, 3
            const uint32_t t = prmt(lo * 3u, hi * 3u, 0x7351u);  // trits of bytes 0..3, one per byte
            w[2 * k] = prmt(ta, tb, t * 0x22u + 0x1010u);
            w[2 * k + 1] = prmt(ta, tb, (t >> 16) * 0x22u + 0x1010u);
        }
    }
};



// gguf:tq2_0: y[j] = M(d, v[j] - 1), v = P(q,2,32) (q at byte 0, d at 64).
template <>
struct Fmt<KF_TQ2_0> {
    static constexpr int B = 256, S = 66, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u;
        const float d = h2f(lds_2<PH>(in, off + 64u));
        const uint4 n = plane2_16(lds_16<false>(in, off + 32u * (cc >> 3) + 16u * (cc & 1u)), (cc >> 1) & 3u);
        const float bias = 8388609.0f;  // 2^23 + 1
        mul4(d, n.x, bias, v);
        mul4(d, n.y, bias, v + 4);
        mul4(d, n.z, bias, v + 8);
        mul4(d, n.w, bias, v + 12);
    }
};

// gguf:q1_0: y[j] = d if bit(q[floor(j/8)], j mod 8) else -d (no multiply).
template <>
struct Fmt<KF_Q1_0> {
    static constexpr int B = 128, S = 18, CE = 16, CPB = 8;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 3) * S;
        const float d = h2f(lds_2<PH>(in, off)), nd = -d;
        const uint32_t bits = lds_2<PH>(in, off + 2u + 2u * (c & 7u));
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = ((bits >> i) & 1u) ? d : nd;
    }
};

// gguf:q2_0: y[j] = M(d, v[j] - 1), v = P(q,2,1): element j is bits 2*(j mod 4)
// of byte floor(j/4), i.e. bits 2i of the chunk's 4 bytes.
template <>
struct Fmt<KF_Q2_0> {
    static constexpr int B = 64, S = 18, CE = 16, CPB = 4;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 2) * S;
        const float d = h2f(lds_2<PH>(in, off));
        const uint32_t w = lds_4(in, off + 2u + 4u * (c & 3u));
        const float bias = 8388609.0f;  // 2^23 + 1
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = __fmul_rn(d, __fsub_rn(__uint_as_float(0x4B000000u | ((w >> (2 * i)) & 3u)), bias));
    }
};

// ---------------------------------------------------------------------------
// IQ2, IQ3 and IQ1 formats ("Mathematical decoding rules", "IQ2, IQ3, and IQ1
// formats").  A block is 8 groups g of 4 lanes l; lane i = 4g + l gives
// outputs 8i..8i+7, so chunk cc (16 outputs) is lanes 2cc and 2cc+1 of group
// cc>>1.  Codebook rows are read from the device copy of the codebooks
// through the read-only cache.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint2 ldg_row8(const uint64_t* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }

// SP(v): the low seven bits of v, completed by their parity as bit 7.
__device__ __forceinline__ uint32_t sp_signs(uint32_t v7) { return v7 | ((__popc(v7) & 1u) << 7); }

// Four outputs M(M(c, v), s) from codebook bytes w (value j in byte j) and
// sign bits sg (bit j set: s = -1).  With s = +-1 the outer product only sets
// the sign, so it is applied to the sign bit of M(c, v).
__device__ __forceinline__ void signed4(float c, uint32_t w, uint32_t sg, float* v) {
    const float z = 8388608.0f;  // 2^23
    v[0] = __uint_as_float(__float_as_uint(__fmul_rn(c, byte_minus<0>(w, z))) ^ ((sg << 31) & 0x80000000u));
    v[1] = __uint_as_float(__float_as_uint(__fmul_rn(c, byte_minus<1>(w, z))) ^ ((sg << 30) & 0x80000000u));
    v[2] = __uint_as_float(__float_as_uint(__fmul_rn(c, byte_minus<2>(w, z))) ^ ((sg << 29) & 0x80000000u));
    v[3] = __uint_as_float(__float_as_uint(__fmul_rn(c, byte_minus<3>(w, z))) ^ ((sg << 28) & 0x80000000u));
}

__device__ __forceinline__ void lane8_signed(float c, uint2 row, uint32_t sg, float* v) {
    signed4(c, row.x, sg, v);
    signed4(c, row.y, sg >> 4, v + 4);
}

// IQ1 lane: y[j] = M(c, A(v[j], delta)) with v = stored/8 - 1 and
// delta = +-1/8.  8*A(v, delta) = stored - (8 -+ 1) is an exact integer, and
// M(c, x) = M(c/8, 8x) exactly (c/8 is exact: c is a binary16 scale times an
// odd integer), so y = M(c8, stored - bias) with bias = 2^23 + 7 or 2^23 + 9.
__device__ __forceinline__ void lane8_shifted(float c8, uint2 row, float bias, float* v) {
    mul4(c8, row.x, bias, v);
    mul4(c8, row.y, bias, v + 4);
}

// c = M(M(d, 0.5 + t), q) of IQ2_XXS / IQ2_XS / IQ2_S (q = 1/4) and IQ3_XXS
// (q = 1/2).
__device__ __forceinline__ float iq_half_scale(float d, uint32_t t, float q) {
    return __fmul_rn(__fmul_rn(d, __fadd_rn(0.5f, static_cast<float>(t))), q);
}

// gguf:iq2_xxs: a = U(b[6+8g:10+8g]); v = G(iq2xxs_grid, b[2+8g+l]),
// s = SP(field(a,7l,7)), c = M(M(d, 0.5 + a>>28), 0.25).
template <>
struct Fmt<KF_IQ2_XXS> {
    static constexpr int B = 256, S = 66, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, g = cc >> 1, l0 = 2u * (cc & 1u);
        const float d = h2f(lds_2<PH>(in, off));
        const uint32_t idx = lds_2<PH>(in, off + 2u + 8u * g + l0);
        const uint32_t a = lds_4(in, off + 6u + 8u * g);
        const float cs = iq_half_scale(d, a >> 28, 0.25f);
        const uint64_t* G = x.grids->iq2xxs;
        lane8_signed(cs, ldg_row8(G + (idx & 255u)), sp_signs((a >> (7u * l0)) & 127u), v);
        lane8_signed(cs, ldg_row8(G + (idx >> 8)), sp_signs((a >> (7u * l0 + 7u)) & 127u), v + 8);
    }
};

// gguf:iq2_xs: a = U(b[2+2i:4+2i]), t = field(b[66+g], 4*floor(l/2), 4);
// v = G(iq2xs_grid, a mod 512), s = SP(floor(a/512)), c = M(M(d, 0.5+t), 0.25).
template <>
struct Fmt<KF_IQ2_XS> {
    static constexpr int B = 256, S = 74, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, g = cc >> 1;
        const float d = h2f(lds_2<PH>(in, off));
        const uint32_t qa = lds_4(in, off + 2u + 4u * cc);
        const uint32_t t = (in[off + 66u + g] >> (4u * (cc & 1u))) & 15u;
        const float cs = iq_half_scale(d, t, 0.25f);
        const uint64_t* G = x.grids->iq2xs;
        lane8_signed(cs, ldg_row8(G + (qa & 511u)), sp_signs((qa >> 9) & 127u), v);
        lane8_signed(cs, ldg_row8(G + ((qa >> 16) & 511u)), sp_signs(qa >> 25), v + 8);
    }
};

// gguf:iq2_s: r = b[2+i] + 256*field(b[66+g], 2l, 2), t = field(b[74+g],
// 4*floor(l/2), 4); v = G(iq2s_grid, r), s = S(b[34+i]), c = M(M(d,0.5+t),0.25).
template <>
struct Fmt<KF_IQ2_S> {
    static constexpr int B = 256, S = 82, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, g = cc >> 1, l0 = 2u * (cc & 1u);
        const float d = h2f(lds_2<PH>(in, off));
        const uint32_t qs = lds_2<PH>(in, off + 2u + 2u * cc);
        const uint32_t qh = in[off + 66u + g] >> (2u * l0);
        const uint32_t t = (in[off + 74u + g] >> (4u * (cc & 1u))) & 15u;
        const uint32_t sg = lds_2<PH>(in, off + 34u + 2u * cc);
        const float cs = iq_half_scale(d, t, 0.25f);
        const uint64_t* G = x.grids->iq2s;
        lane8_signed(cs, ldg_row8(G + ((qs & 255u) | ((qh & 3u) << 8))), sg & 255u, v);
        lane8_signed(cs, ldg_row8(G + ((qs >> 8) | (((qh >> 2) & 3u) << 8))), sg >> 8, v + 8);
    }
};

// gguf:iq3_xxs: a = U(b[66+4g:70+4g]); v = G(iq3xxs_grid, b[2+2i]) followed
// by G(iq3xxs_grid, b[3+2i]), s = SP(field(a,7l,7)), c = M(M(d, 0.5 + a>>28), 0.5).
template <>
struct Fmt<KF_IQ3_XXS> {
    static constexpr int B = 256, S = 98, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, g = cc >> 1, l0 = 2u * (cc & 1u);
        const float d = h2f(lds_2<PH>(in, off));
        const uint32_t q = lds_4(in, off + 2u + 4u * cc);
        const uint32_t a = lds_4(in, off + 66u + 4u * g);
        const float cs = iq_half_scale(d, a >> 28, 0.5f);
        const uint32_t* G = x.grids->iq3xxs;
        const uint2 r0 = make_uint2(__ldg(G + (q & 255u)), __ldg(G + ((q >> 8) & 255u)));
        const uint2 r1 = make_uint2(__ldg(G + ((q >> 16) & 255u)), __ldg(G + (q >> 24)));
        lane8_signed(cs, r0, sp_signs((a >> (7u * l0)) & 127u), v);
        lane8_signed(cs, r1, sp_signs((a >> (7u * l0 + 7u)) & 127u), v + 8);
    }
};

// gguf:iq3_s: r[t] = b[2+2i+t] + 256*bit(b[66+g], 2l+t); v = G(iq3s_grid,
// r[0]) followed by G(iq3s_grid, r[1]), s = S(b[74+i]),
// c = M(d, 1 + 2*field(b[106+floor(g/2)], 4*(g mod 2), 4)).
template <>
struct Fmt<KF_IQ3_S> {
    static constexpr int B = 256, S = 110, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, g = cc >> 1, l0 = 2u * (cc & 1u);
        const float d = h2f(lds_2<PH>(in, off));
        const uint32_t q = lds_4(in, off + 2u + 4u * cc);
        const uint32_t qh = in[off + 66u + g] >> (2u * l0);  // bits t, lane order: r0, r1, r0', r1'
        const uint32_t sg = lds_2<PH>(in, off + 74u + 2u * cc);
        const uint32_t sc = (in[off + 106u + (g >> 1)] >> (4u * (g & 1u))) & 15u;
        const float cs = __fmul_rn(d, static_cast<float>(1u + 2u * sc));
        const uint32_t* G = x.grids->iq3s;
        const uint2 r0 = make_uint2(__ldg(G + ((q & 255u) | ((qh & 1u) << 8))),
                                    __ldg(G + (((q >> 8) & 255u) | (((qh >> 1) & 1u) << 8))));
        const uint2 r1 = make_uint2(__ldg(G + (((q >> 16) & 255u) | (((qh >> 2) & 1u) << 8))),
                                    __ldg(G + ((q >> 24) | (((qh >> 3) & 1u) << 8))));
        lane8_signed(cs, r0, sg & 255u, v);
        lane8_signed(cs, r1, sg >> 8, v + 8);
    }
};

// gguf:iq1_s: a = U(b[34+2g:36+2g]), r = b[2+i] + 256*field(a,3l,3),
// c = M(d, 2*field(a,12,3)+1), delta = -1/8 if bit(a,15) else 1/8;
// y = M(c, A(G(iq1s_grid, r)[j], delta)).
template <>
struct Fmt<KF_IQ1_S> {
    static constexpr int B = 256, S = 50, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, g = cc >> 1, l0 = 2u * (cc & 1u);
        const float d = h2f(lds_2<PH>(in, off));
        const uint32_t qs = lds_2<PH>(in, off + 2u + 2u * cc);
        const uint32_t a = lds_2<PH>(in, off + 34u + 2u * g);
        const float c8 = __fmul_rn(__fmul_rn(d, static_cast<float>(2u * ((a >> 12) & 7u) + 1u)), 0.125f);
        const float bias = (a >> 15) ? 8388617.0f : 8388615.0f;  // 2^23 + 9 / 2^23 + 7
        const uint32_t hi = a >> (3u * l0);
        const uint64_t* G = x.grids->iq1s;
        lane8_shifted(c8, ldg_row8(G + ((qs & 255u) | ((hi & 7u) << 8))), bias, v);
        lane8_shifted(c8, ldg_row8(G + ((qs >> 8) | (((hi >> 3) & 7u) << 8))), bias, v + 8);
    }
};

// gguf:iq1_m: w[k] = U(b[48+2k:50+2k]); d is the binary16 whose nibble k is
// floor(w[k]/2^12); a = field(b[32+floor(i/2)], 4*(i mod 2), 4),
// r = b[i] + 256*(a mod 8), t = field(w[floor(g/2)], 6*(g mod 2)+3*floor(l/2), 3),
// c = M(d, 2t+1), delta = -1/8 if bit(a,3) else 1/8.
template <>
struct Fmt<KF_IQ1_M> {
    static constexpr int B = 256, S = 56, CE = 16, CPB = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint32_t off = ph + (c >> 4) * S, cc = c & 15u, g = cc >> 1;
        const uint2 w = lds_8(in, off + 48u);  // w[0] | w[1] << 16, w[2] | w[3] << 16
        const uint32_t hb = ((w.x >> 12) & 0x000Fu) | ((w.x >> 24) & 0x00F0u) | ((w.y >> 4) & 0x0F00u) |
                            ((w.y >> 16) & 0xF000u);
        const float d = h2f(hb);
        const uint32_t ww = (g & 4u) ? w.y : w.x;  // holds w[floor(g/2)] in its half (g>>1)&1
        const uint32_t t = (ww >> (16u * ((g >> 1) & 1u) + 6u * (g & 1u) + 3u * (cc & 1u))) & 7u;
        const float c8 = __fmul_rn(__fmul_rn(d, static_cast<float>(2u * t + 1u)), 0.125f);
        const uint32_t qs = lds_2<PH>(in, off + 2u * cc);
        const uint32_t qh = in[off + 32u + cc];
        const uint64_t* G = x.grids->iq1s;
        lane8_shifted(c8, ldg_row8(G + ((qs & 255u) | ((qh & 7u) << 8))), (qh & 8u) ? 8388617.0f : 8388615.0f, v);
        lane8_shifted(c8, ldg_row8(G + ((qs >> 8) | (((qh >> 4) & 7u) << 8))), (qh & 128u) ? 8388617.0f : 8388615.0f,
                      v + 8);
    }
};

// ---------------------------------------------------------------------------
// NInfer grouped schemes q5_g64_fp16, q6_g64_fp16, t2_g128_fp16 (q2_g64_fp16
// is byte-identical to gguf:q2_0) and the row-scaled FP8 formats
// ("tensor-formats" sections 4-6.2 and fp8_e4m3fn_row_*).  Grouped blocks:
// a binary16 scale, then the codes as an LSB-first bit stream;
// w = binary32(s32 * binary32(q)).
// ---------------------------------------------------------------------------

// 16 codes of W bits from the bit stream held in q (bits [0, 16W)), as
// two's-complement values: v[i] = M(d, q_i).  The word u becomes the float
// 2^23 + (u XOR 2^(W-1)) by one bitwise operation; subtracting 2^23 + 2^(W-1)
// leaves the signed code exactly.
template <int W>
__device__ __forceinline__ void twos16(float d, uint4 q, float* v) {
    const uint32_t w[5] = {q.x, q.y, q.z, q.w, 0u};
    constexpr uint32_t mask = (1u << W) - 1u, flip = 0x4B000000u | (1u << (W - 1));
    constexpr float bias = 8388608.0f + static_cast<float>(1u << (W - 1));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int bit = W * i;
        const uint32_t u = __funnelshift_r(w[bit >> 5], w[(bit >> 5) + 1], bit & 31) & mask;
        v[i] = __fmul_rn(d, __fsub_rn(__uint_as_float(u ^ flip), bias));
    }
}

// q5_g64_fp16 / q6_g64_fp16: B = 64, 4 chunks per block; chunk c&3 holds
// bits [16W*(c&3), 16W*(c&3+1)) of the stream, i.e. 2W bytes at 2 + 2W*(c&3).
template <int W, int S_>
struct GroupedTwos {
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v) {
        const uint32_t off = ph + (c >> 2) * S_;
        const float d = h2f(lds_2<PH>(in, off));
        twos16<W>(d, lds_16<false>(in, off + 2u + 2u * W * (c & 3u)), v);
    }
};
template <>
struct Fmt<KF_Q5_G64> {
    static constexpr int B = 64, S = 42, CE = 16, CPB = 4;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        GroupedTwos<5, 42>::chunk<PH>(in, ph, c, v);
    }
};
template <>
struct Fmt<KF_Q6_G64> {
    static constexpr int B = 64, S = 50, CE = 16, CPB = 4;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        GroupedTwos<6, 50>::chunk<PH>(in, ph, c, v);
    }
};

// t2_g128_fp16: B = 128, 8 chunks per block of 4 code bytes each.
template <>
struct Fmt<KF_T2_G128> {
    static constexpr int B = 128, S = 34, CE = 16, CPB = 8;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx&) {
        const uint32_t off = ph + (c >> 3) * S;
        const float d = h2f(lds_2<PH>(in, off));
        twos16<2>(d, make_uint4(lds_4(in, off + 2u + 4u * (c & 7u)), 0u, 0u, 0u), v);
    }
};

// E4M3FN word to binary32 (bias 7; 0x7f / 0xff NaN; sign on every word):
// the exponent and fraction bits placed at binary32's fraction top give
// 2^(e-127)(1+m/8) (or m*2^-129 for e = 0), and the exact factor 2^120
// rebiases them to 2^(e-7)(1+m/8) (or m*2^-9).
__device__ __forceinline__ float e4m3fn_word(uint32_t b) {
    const float m = __fmul_rn(__uint_as_float(((b & 0x7Fu) << 20) | ((b & 0x80u) << 24)), 0x1p120f);
    return ((b & 0x7Fu) == 0x7Fu) ? __uint_as_float(0x7FC00000u) : m;
}

// Row multiplier `row` of an fp8 row tensor (16-bit little-endian words,
// any alignment): BF16 (the high half of a binary32) or binary16.
template <bool BF>
__device__ __forceinline__ float row_multiplier(const uint8_t* plane, uint64_t row) {
    const uint8_t* p = plane + 2u * row;
    const uint32_t w = static_cast<uint32_t>(__ldg(p)) | (static_cast<uint32_t>(__ldg(p + 1)) << 8);
    return BF ? __uint_as_float(w << 16) : h2f(w);
}

// fp8_e4m3fn_row_*: the kernel sees 16-code units (B = S = 16); y = M(c32, s32)
// with s32 the multiplier of the code's row (element e is in row e / K).
template <bool BF>
struct Fp8Row {
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v,
                                                 const Ctx& x) {
        const uint4 q = lds_16<!PH>(in, ph + 16u * c);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        const uint64_t K = x.blocks_per_div;
        const uint64_t e0 = (x.block0 + c) * 16u;
        // row and column from the tile's first code (row0, col0): the offset
        // exceeds K only by a few rows, found by a 32-bit division when
        // everything fits in 32 bits
        uint64_t row = x.row0, col = x.col0 + 16u * c;
        if (col >= K) {
            const uint64_t q = ((col | K) >> 32) == 0 ? static_cast<uint64_t>(static_cast<uint32_t>(col) /
                                                                             static_cast<uint32_t>(K))
                                                      : col / K;
            row += q;
            col -= q * K;
        }
        float s = row_multiplier<BF>(x.divs, row);
        if (col + 16u <= K) {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(e4m3fn_word((w[i >> 2] >> (8 * (i & 3))) & 255u), s);
        } else {
            // the unit crosses a row boundary (K not a multiple of 16)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (col == K) {
                    ++row;
                    col = 0;
                    if (e0 + i < x.n_el) s = row_multiplier<BF>(x.divs, row);
                }
                v[i] = __fmul_rn(e4m3fn_word((w[i >> 2] >> (8 * (i & 3))) & 255u), s);
                ++col;
            }
        }
    }
    // The same unit as 16-bit outputs of type O (pairs in w[0..7]).  Every
    // E4M3FN word, NaN included, is exactly a binary16 value, so the
    // hardware pair conversion gives the code's value; its binary32 product
    // with the multiplier is then rounded once, as above.  A unit that
    // crosses a row boundary takes the element-wise form.
    template <bool PH, int O>
    __device__ __forceinline__ static void chunk16(const uint8_t* in, uint32_t ph, uint32_t c, uint32_t* w,
                                                   const Ctx& x) {
        const uint64_t K = x.blocks_per_div;
        uint64_t row = x.row0, col = x.col0 + 16u * c;
        if (col >= K) {
            const uint64_t q = ((col | K) >> 32) == 0 ? static_cast<uint64_t>(static_cast<uint32_t>(col) /
                                                                             static_cast<uint32_t>(K))
                                                      : col / K;
            row += q;
            col -= q * K;
        }
        if (col + 16u > K) {
            float v[16];
            chunk<PH>(in, ph, c, v, x);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                w[i] = (O == KO_BF16) ? pack_bf16(v[2 * i], v[2 * i + 1]) : pack_f16(v[2 * i], v[2 * i + 1]);
            return;
        }
        const uint4 q = lds_16<!PH>(in, ph + 16u * c);
        const uint32_t cw[4] = {q.x, q.y, q.z, q.w};
        const float s = row_multiplier<BF>(x.divs, row);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>((cw[i >> 1] >> (16 * (i & 1))) & 0xffffu), __NV_E4M3);
            const float a = __fmul_rn(__half2float(__ushort_as_half(h.x)), s);
            const float b = __fmul_rn(__half2float(__ushort_as_half(h.y)), s);
            w[i] = (O == KO_BF16) ? pack_bf16(a, b) : pack_f16(a, b);
        }
    }
};
template <>
struct Fmt<KF_FP8_ROW_BF16> {
    static constexpr int B = 16, S = 16, CE = 16, CPB = 1;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx& x) {
        Fp8Row<true>::chunk<PH>(in, ph, c, v, x);
    }
    template <bool PH, int O>
    __device__ __forceinline__ static void chunk16(const uint8_t* in, uint32_t ph, uint32_t c, uint32_t* w,
                                                   const Ctx& x) {
        Fp8Row<true>::template chunk16<PH, O>(in, ph, c, w, x);
    }
};
template <>
struct Fmt<KF_FP8_ROW_FP16> {
    static constexpr int B = 16, S = 16, CE = 16, CPB = 1;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, float* v, const Ctx& x) {
        Fp8Row<false>::chunk<PH>(in, ph, c, v, x);
    }
    template <bool PH, int O>
    __device__ __forceinline__ static void chunk16(const uint8_t* in, uint32_t ph, uint32_t c, uint32_t* w,
                                                   const Ctx& x) {
        Fp8Row<false>::template chunk16<PH, O>(in, ph, c, w, x);
    }
};

// Decoders that decode a lane's two 8-element runs of a pair of adjacent
// chunks lying in one block (pair_runs): each of the pair's two store
// instructions then fills a whole 32-byte sector without any exchange between
// the lanes.  (q4_k and q8_0 measured slower this way than with the exchange
// of store16_pairs; q6_k faster.)
template <int F>
struct has_pair_runs {
    static constexpr bool value = F == KF_Q6_K;
};

// Decoders that also produce 16-bit outputs directly (chunk16).
template <int F>
struct has_chunk16 {
    static constexpr bool value = F == KF_TQ1_0 || F == KF_FP8_ROW_BF16 || F == KF_FP8_ROW_FP16;
};

// ---------------------------------------------------------------------------
// Output stage: one RNE conversion per element; 16-byte stores when y is
// 16-byte aligned (chunk offsets are multiples of 8 elements, so every chunk
// then starts on a 16-byte boundary).
// ---------------------------------------------------------------------------

template <int O, int N>
__device__ __forceinline__ void store_chunk(void* y, uint64_t e0, const float* v, bool vec) {
    if (O == KO_F32) {
        float* p = static_cast<float*>(y) + e0;
        if (vec) {
#pragma unroll
            for (int i = 0; i < N / 4; ++i)
                reinterpret_cast<float4*>(p)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) p[i] = v[i];
        }
    } else if (O == KO_F64) {
        double* p = static_cast<double*>(y) + e0;
        if (vec) {
#pragma unroll
            for (int i = 0; i < N / 2; ++i)
                reinterpret_cast<double2*>(p)[i] =
                    make_double2(static_cast<double>(v[2 * i]), static_cast<double>(v[2 * i + 1]));
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) p[i] = static_cast<double>(v[i]);
        }
    } else {
        uint32_t w[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i)
            w[i] = (O == KO_BF16) ? pack_bf16(v[2 * i], v[2 * i + 1]) : pack_f16(v[2 * i], v[2 * i + 1]);
        uint16_t* p = static_cast<uint16_t*>(y) + e0;
        if (vec) {
#pragma unroll
            for (int i = 0; i < N / 8; ++i)
                reinterpret_cast<uint4*>(p)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                p[2 * i] = static_cast<uint16_t>(w[i] & 0xffffu);
                p[2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
            }
        }
    }
}

// The last 16 codes of an fp8 row tensor may be fewer than 16: one scalar
// store per valid element.
template <int O>
__device__ __forceinline__ void store_partial(void* y, uint64_t e0, const float* v, uint32_t n) {
    for (uint32_t i = 0; i < n; ++i) {
        if (O == KO_F32) static_cast<float*>(y)[e0 + i] = v[i];
        else if (O == KO_F64) static_cast<double*>(y)[e0 + i] = static_cast<double>(v[i]);
        else if (O == KO_BF16) static_cast<__nv_bfloat16*>(y)[e0 + i] = __float2bfloat16_rn(v[i]);
        else static_cast<__half*>(y)[e0 + i] = __float2half_rn(v[i]);
    }
}

// ---------------------------------------------------------------------------
// Byte-table decode of nvfp4 to a 16-bit output.  The output of an element
// depends only on its group's scale byte s, its 4-bit code c and the tile's
// divisor, so each CTA tabulates the 16-bit result of (s, c) for the codes
// c < 8 once, computed by the format's own rule (one division) and cast
// once: row s (16 bytes) holds their high bytes, then their low bytes.  A
// code c | 8 decodes to the negated value of c: E2M1 word 8 + m is
// -e2m1(m) (word 8 is -0), the product with the scale is exact, and RNE
// division and the RNE cast are odd-symmetric.  Decoding is then pure data
// movement: one prmt looks up 4 codes' high (or low) bytes in the row, the
// sign bit is flipped from each code's bit 3, and two more prmts pair low
// and high bytes into output words.
// ---------------------------------------------------------------------------
// The table for divisor dw and output type O (row s in words 4s..4s+3 of
// L), written by threads tid, tid + nthr, ...
template <int O>
__device__ __forceinline__ void build_lut16(uint32_t* L, float dw, uint32_t tid, uint32_t nthr) {
    for (uint32_t i = tid; i < 512u; i += nthr) {
        const uint32_t s = i >> 1, c0 = 4u * (i & 1u);
        uint32_t hi = 0, lo = 0;
#pragma unroll
        for (uint32_t j = 0; j < 4; ++j) {
            const uint32_t c = c0 + j;
            const float w = __fdiv_rn(__fmul_rn(e2m1(c), e4m3fn(s)), dw);
            const uint32_t h = (O == KO_BF16) ? (pack_bf16(w, 0.0f) & 0xffffu) : (pack_f16(w, 0.0f) & 0xffffu);
            hi |= (h >> 8) << (8u * j);
            lo |= (h & 0xffu) << (8u * j);
        }
        L[4u * s + (i & 1u)] = hi;
        L[4u * s + 2u + (i & 1u)] = lo;
    }
}

// Eight codes (the nibbles of q, low nibble first) through table row r.
// The nibbles of q are codes of elements e0, f0, e1, f1, e2, f2, e3, f3,
// where e and f are two runs of 4 consecutive outputs: a0 and a1 receive
// (e0, e1) and (e2, e3), b0 and b1 receive (f0, f1) and (f2, f3), as pairs
// of 16-bit words (the first element in the low half).
__device__ __forceinline__ void lut16_word(uint32_t q, uint4 r, uint32_t& a0, uint32_t& a1, uint32_t& b0, uint32_t& b1) {
    // 0x80 in output byte i where the code in selector nibble i has bit 3
    // set: prmt's sign-replicating selectors copy the top bit of a source
    // byte, and the top bits of q << 4 and q are the codes' bit 3.
    const uint32_t t = q << 4;
    const uint32_t ma = prmt(t, q, 0xD9C8u) & 0x80808080u, mb = prmt(t, q, 0xFBEAu) & 0x80808080u;
    const uint32_t sa = q & 0x7777u, sb = (q >> 16) & 0x7777u;  // codes mod 8
    uint32_t h = prmt(r.x, r.y, sa) ^ ma, l = prmt(r.z, r.w, sa);
    a0 = prmt(l, h, 0x6240u);
    b0 = prmt(l, h, 0x7351u);
    h = prmt(r.x, r.y, sb) ^ mb;
    l = prmt(r.z, r.w, sb);
    a1 = prmt(l, h, 0x6240u);
    b1 = prmt(l, h, 0x7351u);
}

template <int N>
__device__ __forceinline__ void store_words16(uint16_t* p, const uint32_t* w, bool vec) {
    if (vec) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i) reinterpret_cast<uint4*>(p)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            p[2 * i] = static_cast<uint16_t>(w[i] & 0xffffu);
            p[2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
        }
    }
}

// Formats whose decode is limited by instruction issue rather than by memory
// (measured): the lane-pair exchange of store16_pairs costs them more than
// whole-sector stores gain.
__host__ __device__ constexpr bool issue_bound(int f) {
    return f == KF_IQ2_XXS || f == KF_IQ2_XS || f == KF_IQ2_S || f == KF_IQ3_XXS || f == KF_IQ3_S || f == KF_IQ1_S ||
           f == KF_IQ1_M;
}

// Stores 16 consecutive 16-bit outputs (words w[0..7]) at element e0 of a
// 16-byte-aligned y.  Every lane of the warp calls it.  When pair_ok, lanes
// 2j and 2j+1 hold adjacent chunks (odd: this lane holds the later one) and
// swap halves so that each store instruction of the pair fills one whole
// 32-byte sector: lane 2j stores bytes [0,16) then [32,48) of the pair's 64
// bytes, lane 2j+1 bytes [16,32) then [48,64).  A lane writing its own 32
// bytes as two 16-byte stores leaves every sector half written per
// instruction, which on GB300 caps the write rate near 3.8 TB/s (6.5 TB/s
// with whole sectors).  Otherwise a lane with ok stores its own chunk.
__device__ __forceinline__ void store16_pairs(uint16_t* y, uint64_t e0, const uint32_t* w, bool odd, bool ok,
                                              bool pair_ok) {
    uint32_t ra[4], rb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        ra[i] = __shfl_xor_sync(0xffffffffu, w[i], 1);
        rb[i] = __shfl_xor_sync(0xffffffffu, w[4 + i], 1);
    }
    if (pair_ok) {
        uint16_t* p = y + e0 - (odd ? 8u : 0u);
        reinterpret_cast<uint4*>(p)[0] = odd ? make_uint4(rb[0], rb[1], rb[2], rb[3]) : make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(p + 16)[0] = odd ? make_uint4(w[4], w[5], w[6], w[7]) : make_uint4(ra[0], ra[1], ra[2], ra[3]);
    } else if (ok) {
        reinterpret_cast<uint4*>(y + e0)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(y + e0)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// Chunk c (16 outputs) of a 16-byte-aligned nvfp4 stage through the table
// (row s at L[s]), as 8 words of output pairs: group g = c & 3 of block
// c >> 2 is its scale byte, then 8 code bytes whose low nibbles are outputs
// 0..7 and high nibbles outputs 8..15 (the blocks' 36-byte stride keeps them
// 4-byte aligned).
__device__ __forceinline__ void lut16_chunk(const uint8_t* in, const uint4* L, uint32_t c, uint32_t* w) {
    const uint32_t off = (c >> 2) * 36u, g = c & 3u;
    const uint32_t s = in[off + g];
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(in + off + 4u + 8u * g);
    const uint4 r = L[s];
    lut16_word(qw[0], r, w[0], w[1], w[4], w[5]);
    lut16_word(qw[1], r, w[2], w[3], w[6], w[7]);
}

// A 16-byte-aligned nvfp4 stage through the table, every consumer thread
// storing its chunks itself.
__device__ __forceinline__ void decode_tile_lut16(const StageInfo& si, const uint8_t* in, const uint4* L, uint32_t tid) {
    uint16_t* y = static_cast<uint16_t*>(si.t.y);
    const bool vec = si.t.yvec != 0;
    const uint32_t nch = si.nb * 4u;
#pragma unroll
    for (int k = 0; k < kTileElems / 16 / kThreads; ++k) {
        const uint32_t c = tid + static_cast<uint32_t>(k * kThreads);
        const bool ok = c < nch;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (ok) lut16_chunk(in, L, c, w);
        const uint64_t e0 = si.block0 * 64u + 16u * c;
        if (vec)  // (uniform over the warp)
            store16_pairs(y, e0, w, c & 1u, ok, (c | 1u) < nch);
        else if (ok)
            store_words16<8>(y + e0, w, false);
    }
}

// Chunk c of a 16-byte-aligned stage as CE/2 words of 16-bit output pairs of
// type O (LUT: the nvfp4 byte table L).
template <int F, int O, bool LUT>
__device__ __forceinline__ void chunk_words(const uint8_t* in, uint32_t c, const Ctx& x, const uint4* L, uint32_t* w) {
    using Fm = Fmt<F>;
    if constexpr (LUT) {
        lut16_chunk(in, L, c, w);
    } else if constexpr (has_chunk16<F>::value) {
        Fm::template chunk16<false, O>(in, 0u, c, w, x);
    } else {
        float v[Fm::CE];
        Fm::template chunk<false>(in, 0u, c, v, x);
#pragma unroll
        for (int i = 0; i < Fm::CE / 2; ++i)
            w[i] = (O == KO_BF16) ? pack_bf16(v[2 * i], v[2 * i + 1]) : pack_f16(v[2 * i], v[2 * i + 1]);
    }
}

// One consumer warp's share of a full, 16-byte-aligned stage with a 16-bit
// output: the warp's kWarpOut consecutive outputs (chunks cw0 + 32k +
// lane), written in output order to the warp's output buffer `ob`, which the
// caller copies to y with one bulk copy.  Chunk j of the share is bytes
// [2*CE*j, 2*CE*(j+1)) of the buffer.
template <int F, int O, bool LUT>
__device__ __forceinline__ void decode_warp16(const uint8_t* in, const Ctx& x, const uint4* L, uint32_t warp,
                                              uint32_t lane, uint8_t* ob) {
    constexpr int CE = LUT ? 16 : Fmt<F>::CE;
    constexpr int kPer = kWarpOut / CE / 32;  // chunks per lane
    const uint32_t cw0 = warp * static_cast<uint32_t>(kWarpOut / CE);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const uint32_t j = static_cast<uint32_t>(32 * k) + lane;
        uint32_t w[CE / 2];
        chunk_words<F, O, LUT>(in, cw0 + j, x, L, w);
        uint4* d = reinterpret_cast<uint4*>(ob) + j * static_cast<uint32_t>(CE / 8);
#pragma unroll
        for (int q = 0; q < CE / 8; ++q) d[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
}

// Output type dispatch (OSEL < 0: the tensor's own 16-bit type).
template <int F, int OSEL, bool LUT>
__device__ __forceinline__ void decode_warp16_o(const StageInfo& si, const uint8_t* in, const Ctx& x, const uint4* L,
                                                uint32_t warp, uint32_t lane, uint8_t* ob) {
    if constexpr (OSEL == KO_F16) {
        decode_warp16<F, KO_F16, LUT>(in, x, L, warp, lane, ob);
    } else if constexpr (OSEL == KO_BF16) {
        decode_warp16<F, KO_BF16, LUT>(in, x, L, warp, lane, ob);
    } else if constexpr (OSEL < 0) {
        if (si.t.out == KO_F16)
            decode_warp16<F, KO_F16, false>(in, x, L, warp, lane, ob);
        else
            decode_warp16<F, KO_BF16, false>(in, x, L, warp, lane, ob);
    }
}

// Format dispatch of a staged warp share (FSEL / OSEL as for k_decode).
template <int FSEL, int OSEL>
__device__ __forceinline__ void decode_warp16_fast(const StageInfo& si, const uint8_t* in, const Ctx& x,
                                                   const uint4* L, uint32_t warp, uint32_t lane, uint8_t* ob) {
    if constexpr (FSEL >= 0) {
        decode_warp16_o<FSEL, OSEL, uses_lut16(FSEL, OSEL)>(si, in, x, L, warp, lane, ob);
    } else if constexpr (FSEL == kFselKQuantMix) {
        switch (si.t.fmt) {
            case KF_Q8_0: decode_warp16_o<KF_Q8_0, OSEL, false>(si, in, x, L, warp, lane, ob); break;
            case KF_Q4_K: decode_warp16_o<KF_Q4_K, OSEL, false>(si, in, x, L, warp, lane, ob); break;
            default: decode_warp16_o<KF_Q6_K, OSEL, false>(si, in, x, L, warp, lane, ob); break;
        }
    } else {
        switch (si.t.fmt) {
#define NDQ_W16(K) \
    case K: decode_warp16_o<K, OSEL, false>(si, in, x, L, warp, lane, ob); break;
            NDQ_W16(KF_Q8_0) NDQ_W16(KF_Q4_0) NDQ_W16(KF_IQ4_NL) NDQ_W16(KF_Q4_K) NDQ_W16(KF_Q6_K)
            NDQ_W16(KF_MXFP4) NDQ_W16(KF_GGUF_NVFP4) NDQ_W16(KF_NVFP4) NDQ_W16(KF_Q4_1) NDQ_W16(KF_Q5_0)
            NDQ_W16(KF_Q5_1) NDQ_W16(KF_Q8_1) NDQ_W16(KF_Q8_K) NDQ_W16(KF_Q2_K) NDQ_W16(KF_Q3_K) NDQ_W16(KF_Q5_K)
            NDQ_W16(KF_IQ4_XS) NDQ_W16(KF_TQ1_0) NDQ_W16(KF_TQ2_0) NDQ_W16(KF_Q1_0) NDQ_W16(KF_Q2_0)
            NDQ_W16(KF_IQ2_XXS) NDQ_W16(KF_IQ2_XS) NDQ_W16(KF_IQ2_S) NDQ_W16(KF_IQ3_XXS) NDQ_W16(KF_IQ3_S)
            NDQ_W16(KF_IQ1_S) NDQ_W16(KF_IQ1_M) NDQ_W16(KF_Q5_G64) NDQ_W16(KF_Q6_G64) NDQ_W16(KF_T2_G128)
            NDQ_W16(KF_FP8_ROW_BF16) NDQ_W16(KF_FP8_ROW_FP16)
#undef NDQ_W16
            default: decode_warp16_o<KF_Q4_G64, OSEL, false>(si, in, x, L, warp, lane, ob); break;
        }
    }
}

template <int F, int O, bool PH>
__device__ __forceinline__ void decode_tile_fop(const StageInfo& si, const uint8_t* in, const Ctx& x, uint32_t tid) {
    using Fm = Fmt<F>;
    const uint32_t nch = si.nb * static_cast<uint32_t>(Fm::CPB);
    const uint64_t e_base = si.block0 * static_cast<uint64_t>(Fm::B);
    const bool vec = si.t.yvec != 0;
    void* y = si.t.y;
    const uint32_t ph = PH ? si.phase : 0u;
    constexpr int kPerThread = kTileElems / Fm::CE / kThreads;  // chunks per thread per tile
    constexpr bool kPair = (O == KO_BF16 || O == KO_F16) && Fm::CE == 16 && !issue_bound(F);
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const uint32_t c = tid + static_cast<uint32_t>(k * kThreads);
        if constexpr (has_pair_runs<F>::value && kPair) {
            if (vec) {
                // lane h of a pair stores pair elements 8h.. and then 24-8h..:
                // both store instructions of the pair fill whole sectors
                if (c < nch) {
                    float v[16];
                    Fm::template pair_runs<PH>(in, ph, c, v, x);
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        w[i] = (O == KO_BF16) ? pack_bf16(v[2 * i], v[2 * i + 1]) : pack_f16(v[2 * i], v[2 * i + 1]);
                    uint16_t* pp = static_cast<uint16_t*>(y) + e_base + 16ull * (c & ~1u);
                    const uint32_t h = c & 1u;
                    reinterpret_cast<uint4*>(pp + 8u * h)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    reinterpret_cast<uint4*>(pp + 24u - 8u * h)[0] = make_uint4(w[4], w[5], w[6], w[7]);
                }
            } else if (c < nch) {
                float v[Fm::CE];
                Fm::template chunk<PH>(in, ph, c, v, x);
                store_chunk<O, Fm::CE>(y, e_base + static_cast<uint64_t>(Fm::CE) * c, v, false);
            }
        } else if (kPair && vec) {
            // adjacent lanes hold adjacent chunks: store them as sector pairs
            const bool ok = c < nch;
            float v[16];
            uint32_t w[8];
            if constexpr (has_chunk16<F>::value) {
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = 0u;
                if (ok) Fm::template chunk16<PH, O>(in, ph, c, w, x);
            } else {
                if (ok) {
                    Fm::template chunk<PH>(in, ph, c, v, x);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    w[i] = (O == KO_BF16) ? pack_bf16(v[2 * i], v[2 * i + 1]) : pack_f16(v[2 * i], v[2 * i + 1]);
            }
            const uint32_t cp = c | 1u;  // the later chunk of the pair
            bool pair_ok = cp < nch;
            if (is_fp8_row(F)) pair_ok = pair_ok && e_base + 16ull * cp + 16u <= x.n_el;
            const uint64_t e0 = e_base + 16ull * c;
            const bool part = is_fp8_row(F) && ok && e0 + 16u > x.n_el;  // a partial last fp8 unit
            store16_pairs(static_cast<uint16_t*>(y), e0, w, c & 1u, ok && !part, pair_ok);
            if (part) {
                if constexpr (has_chunk16<F>::value) Fm::template chunk<PH>(in, ph, c, v, x);
                store_partial<O>(y, e0, v, static_cast<uint32_t>(x.n_el - e0));
            }
        } else if (c < nch) {
            float v[Fm::CE];
            Fm::template chunk<PH>(in, ph, c, v, x);
            const uint64_t e0 = e_base + static_cast<uint64_t>(Fm::CE) * c;
            if (is_fp8_row(F) && e0 + Fm::CE > x.n_el)
                store_partial<O>(y, e0, v, static_cast<uint32_t>(x.n_el - e0));
            else
                store_chunk<O, Fm::CE>(y, e0, v, vec);
        }
    }
}

// Slow path, shared by every kernel and never inlined: a stage at a nonzero
// byte phase (an unaligned payload pointer) or an nvfp4 tile whose divisor is
// not the one the shared quotient table holds (per-element division).
template <int F>
__device__ __forceinline__ void decode_tile_slow_f(const StageInfo& si, const uint8_t* in, const Ctx& x,
                                                   uint32_t tid) {
    switch (si.t.out) {
        case KO_F32: decode_tile_fop<F, KO_F32, true>(si, in, x, tid); break;
        case KO_F16: decode_tile_fop<F, KO_F16, true>(si, in, x, tid); break;
        case KO_BF16: decode_tile_fop<F, KO_BF16, true>(si, in, x, tid); break;
        default: decode_tile_fop<F, KO_F64, true>(si, in, x, tid); break;
    }
}

// Slow path of a kernel specialised for format F (and output type O when
// O >= 0): only that decoder, so the specialised kernel's register budget is
// not set by the other formats' slow paths.
template <int F, int O>
__device__ __noinline__ void decode_tile_slow_one(const StageInfo& si, const uint8_t* in, const Ctx x, uint32_t tid) {
    if (O >= 0)
        decode_tile_fop<F, (O >= 0 ? O : 0), true>(si, in, x, tid);
    else
        decode_tile_slow_f<F>(si, in, x, tid);
}

__device__ __noinline__ void decode_tile_slow(const StageInfo& si, const uint8_t* in, const Ctx x, uint32_t tid) {
    switch (si.t.fmt) {
        case KF_Q8_0: decode_tile_slow_f<KF_Q8_0>(si, in, x, tid); break;
        case KF_Q4_0: decode_tile_slow_f<KF_Q4_0>(si, in, x, tid); break;
        case KF_IQ4_NL: decode_tile_slow_f<KF_IQ4_NL>(si, in, x, tid); break;
        case KF_Q4_K: decode_tile_slow_f<KF_Q4_K>(si, in, x, tid); break;
        case KF_Q6_K: decode_tile_slow_f<KF_Q6_K>(si, in, x, tid); break;
        case KF_MXFP4: decode_tile_slow_f<KF_MXFP4>(si, in, x, tid); break;
        case KF_GGUF_NVFP4: decode_tile_slow_f<KF_GGUF_NVFP4>(si, in, x, tid); break;
        case KF_NVFP4: decode_tile_slow_f<KF_NVFP4>(si, in, x, tid); break;
        case KF_Q4_1: decode_tile_slow_f<KF_Q4_1>(si, in, x, tid); break;
        case KF_Q5_0: decode_tile_slow_f<KF_Q5_0>(si, in, x, tid); break;
        case KF_Q5_1: decode_tile_slow_f<KF_Q5_1>(si, in, x, tid); break;
        case KF_Q8_1: decode_tile_slow_f<KF_Q8_1>(si, in, x, tid); break;
        case KF_Q8_K: decode_tile_slow_f<KF_Q8_K>(si, in, x, tid); break;
        case KF_Q2_K: decode_tile_slow_f<KF_Q2_K>(si, in, x, tid); break;
        case KF_Q3_K: decode_tile_slow_f<KF_Q3_K>(si, in, x, tid); break;
        case KF_Q5_K: decode_tile_slow_f<KF_Q5_K>(si, in, x, tid); break;
        case KF_IQ4_XS: decode_tile_slow_f<KF_IQ4_XS>(si, in, x, tid); break;
        case KF_TQ1_0: decode_tile_slow_f<KF_TQ1_0>(si, in, x, tid); break;
        case KF_TQ2_0: decode_tile_slow_f<KF_TQ2_0>(si, in, x, tid); break;
        case KF_Q1_0: decode_tile_slow_f<KF_Q1_0>(si, in, x, tid); break;
        case KF_Q2_0: decode_tile_slow_f<KF_Q2_0>(si, in, x, tid); break;
        case KF_IQ2_XXS: decode_tile_slow_f<KF_IQ2_XXS>(si, in, x, tid); break;
        case KF_IQ2_XS: decode_tile_slow_f<KF_IQ2_XS>(si, in, x, tid); break;
        case KF_IQ2_S: decode_tile_slow_f<KF_IQ2_S>(si, in, x, tid); break;
        case KF_IQ3_XXS: decode_tile_slow_f<KF_IQ3_XXS>(si, in, x, tid); break;
        case KF_IQ3_S: decode_tile_slow_f<KF_IQ3_S>(si, in, x, tid); break;
        case KF_IQ1_S: decode_tile_slow_f<KF_IQ1_S>(si, in, x, tid); break;
        case KF_IQ1_M: decode_tile_slow_f<KF_IQ1_M>(si, in, x, tid); break;
        case KF_Q5_G64: decode_tile_slow_f<KF_Q5_G64>(si, in, x, tid); break;
        case KF_Q6_G64: decode_tile_slow_f<KF_Q6_G64>(si, in, x, tid); break;
        case KF_T2_G128: decode_tile_slow_f<KF_T2_G128>(si, in, x, tid); break;
        case KF_FP8_ROW_BF16: decode_tile_slow_f<KF_FP8_ROW_BF16>(si, in, x, tid); break;
        case KF_FP8_ROW_FP16: decode_tile_slow_f<KF_FP8_ROW_FP16>(si, in, x, tid); break;
        default: decode_tile_slow_f<KF_Q4_G64>(si, in, x, tid); break;
    }
}

// Fast path: 16-byte-aligned stage (and, for nvfp4, the shared table).
// OSEL / FSEL fix the output type / format at compile time, or are -1 for a
// runtime switch (batched launches that mix them).
template <int F, int OSEL>
__device__ __forceinline__ void decode_tile_fast_f(const StageInfo& si, const uint8_t* in, const Ctx& x,
                                                   uint32_t tid) {
    if (OSEL >= 0) {
        decode_tile_fop<F, (OSEL >= 0 ? OSEL : 0), false>(si, in, x, tid);
        return;
    }
    switch (si.t.out) {
        case KO_F32: decode_tile_fop<F, KO_F32, false>(si, in, x, tid); break;
        case KO_F16: decode_tile_fop<F, KO_F16, false>(si, in, x, tid); break;
        case KO_BF16: decode_tile_fop<F, KO_BF16, false>(si, in, x, tid); break;
        default: decode_tile_fop<F, KO_F64, false>(si, in, x, tid); break;
    }
}

template <int FSEL, int OSEL>
__device__ __forceinline__ void decode_tile_fast(const StageInfo& si, const uint8_t* in, const Ctx& x,
                                                 uint32_t tid) {
    if (FSEL >= 0) {
        decode_tile_fast_f<(FSEL >= 0 ? FSEL : 0), OSEL>(si, in, x, tid);
        return;
    }
    if (FSEL == kFselKQuantMix) {  // q8_0 / q4_k / q6_k only (other formats: slow path)
        switch (si.t.fmt) {
            case KF_Q8_0: decode_tile_fast_f<KF_Q8_0, OSEL>(si, in, x, tid); break;
            case KF_Q4_K: decode_tile_fast_f<KF_Q4_K, OSEL>(si, in, x, tid); break;
            case KF_Q6_K: decode_tile_fast_f<KF_Q6_K, OSEL>(si, in, x, tid); break;
            default: decode_tile_slow(si, in, x, tid); break;
        }
        return;
    }
    switch (si.t.fmt) {
        case KF_Q8_0: decode_tile_fast_f<KF_Q8_0, OSEL>(si, in, x, tid); break;
        case KF_Q4_0: decode_tile_fast_f<KF_Q4_0, OSEL>(si, in, x, tid); break;
        case KF_IQ4_NL: decode_tile_fast_f<KF_IQ4_NL, OSEL>(si, in, x, tid); break;
        case KF_Q4_K: decode_tile_fast_f<KF_Q4_K, OSEL>(si, in, x, tid); break;
        case KF_Q6_K: decode_tile_fast_f<KF_Q6_K, OSEL>(si, in, x, tid); break;
        case KF_MXFP4: decode_tile_fast_f<KF_MXFP4, OSEL>(si, in, x, tid); break;
        case KF_GGUF_NVFP4: decode_tile_fast_f<KF_GGUF_NVFP4, OSEL>(si, in, x, tid); break;
        case KF_NVFP4: decode_tile_fast_f<KF_NVFP4, OSEL>(si, in, x, tid); break;
        case KF_Q4_1: decode_tile_fast_f<KF_Q4_1, OSEL>(si, in, x, tid); break;
        case KF_Q5_0: decode_tile_fast_f<KF_Q5_0, OSEL>(si, in, x, tid); break;
        case KF_Q5_1: decode_tile_fast_f<KF_Q5_1, OSEL>(si, in, x, tid); break;
        case KF_Q8_1: decode_tile_fast_f<KF_Q8_1, OSEL>(si, in, x, tid); break;
        case KF_Q8_K: decode_tile_fast_f<KF_Q8_K, OSEL>(si, in, x, tid); break;
        case KF_Q2_K: decode_tile_fast_f<KF_Q2_K, OSEL>(si, in, x, tid); break;
        case KF_Q3_K: decode_tile_fast_f<KF_Q3_K, OSEL>(si, in, x, tid); break;
        case KF_Q5_K: decode_tile_fast_f<KF_Q5_K, OSEL>(si, in, x, tid); break;
        case KF_IQ4_XS: decode_tile_fast_f<KF_IQ4_XS, OSEL>(si, in, x, tid); break;
        case KF_TQ1_0: decode_tile_fast_f<KF_TQ1_0, OSEL>(si, in, x, tid); break;
        case KF_TQ2_0: decode_tile_fast_f<KF_TQ2_0, OSEL>(si, in, x, tid); break;
        case KF_Q1_0: decode_tile_fast_f<KF_Q1_0, OSEL>(si, in, x, tid); break;
        case KF_Q2_0: decode_tile_fast_f<KF_Q2_0, OSEL>(si, in, x, tid); break;
        case KF_IQ2_XXS: decode_tile_fast_f<KF_IQ2_XXS, OSEL>(si, in, x, tid); break;
        case KF_IQ2_XS: decode_tile_fast_f<KF_IQ2_XS, OSEL>(si, in, x, tid); break;
        case KF_IQ2_S: decode_tile_fast_f<KF_IQ2_S, OSEL>(si, in, x, tid); break;
        case KF_IQ3_XXS: decode_tile_fast_f<KF_IQ3_XXS, OSEL>(si, in, x, tid); break;
        case KF_IQ3_S: decode_tile_fast_f<KF_IQ3_S, OSEL>(si, in, x, tid); break;
        case KF_IQ1_S: decode_tile_fast_f<KF_IQ1_S, OSEL>(si, in, x, tid); break;
        case KF_IQ1_M: decode_tile_fast_f<KF_IQ1_M, OSEL>(si, in, x, tid); break;
        case KF_Q5_G64: decode_tile_fast_f<KF_Q5_G64, OSEL>(si, in, x, tid); break;
        case KF_Q6_G64: decode_tile_fast_f<KF_Q6_G64, OSEL>(si, in, x, tid); break;
        case KF_T2_G128: decode_tile_fast_f<KF_T2_G128, OSEL>(si, in, x, tid); break;
        case KF_FP8_ROW_BF16: decode_tile_fast_f<KF_FP8_ROW_BF16, OSEL>(si, in, x, tid); break;
        case KF_FP8_ROW_FP16: decode_tile_fast_f<KF_FP8_ROW_FP16, OSEL>(si, in, x, tid); break;
        default: decode_tile_fast_f<KF_Q4_G64, OSEL>(si, in, x, tid); break;
    }
}

// ---------------------------------------------------------------------------
// Producer warp (lane 0): stages tiles it = 0, 1, ... of this CTA.
// ---------------------------------------------------------------------------
// The payload span of a tile: its first block, block count, source and the
// 16-byte lines holding it (from the line below its first byte to the line
// above its last; an fp8 row tensor's span stops at the end of its code
// plane, before the row multipliers).
struct TileSpan {
    uint64_t b0;
    const uint8_t* src;
    uint32_t nb, phase, bytes;
};
__device__ __forceinline__ TileSpan tile_span(const DevTensor& t, uint64_t tile) {
    TileSpan r;
    r.b0 = (tile - t.tile_begin) * t.bpt;
    const uint64_t left = t.nblocks - r.b0;
    r.nb = left < t.bpt ? static_cast<uint32_t>(left) : t.bpt;
    r.src = t.x + r.b0 * t.S;
    r.phase = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(r.src) & 15u);
    uint32_t span = r.nb * t.S;
    if (t.fmt == KF_FP8_ROW_BF16 || t.fmt == KF_FP8_ROW_FP16) {
        const uint64_t plane = reinterpret_cast<uintptr_t>(t.divs) - reinterpret_cast<uintptr_t>(r.src);
        if (plane < span) span = static_cast<uint32_t>(plane);
    }
    r.bytes = (r.phase + span + 15u) & ~15u;
    return r;
}

template <int NST>
__device__ void producer(const KParams& p, SmemHdr& H, uint8_t* inbuf) {
    static_assert(NST <= kStages, "decode stages");
    const uint64_t grid = gridDim.x;
    int32_t di = 0;   // current tensor (tiles of a CTA increase, so it only moves forward)
    int issued = 0;   // tiles staged so far
    bool fault = false;
    // nvfp4: the last divisor compared with the shared tables' (tensor,
    // index), so that a tile whose divisor was seen before issues no load
    int32_t nv_di = -1;
    uint64_t nv_d = 0;
    uint32_t nv_same = 0;
    int withheld = -1;  // staging whose copy was withheld on request (never completes)
    for (uint64_t tile = blockIdx.x; tile < p.total_tiles; tile += grid, ++issued) {
        const int s = issued % NST;
        if (issued >= NST &&
            !mbar_wait_bounded(&H.empty[s], static_cast<uint32_t>(((issued / NST) - 1) & 1), p.wait_ns)) {
            fault = true;
            break;
        }
        if (static_cast<int64_t>(tile) == p.withhold_tile) {
            // failure-path check requested by the host (ndq_test_withhold_copy):
            // this tile's stage is never filled, so the consumers' bounded
            // wait for it runs out
            withheld = issued;
            continue;
        }
        if (p.table)
            while (di + 1 < p.n && p.table[di + 1].tile_begin <= tile) ++di;
        const DevTensor& t = p.table ? p.table[di] : p.single;
        StageInfo& si = H.info[s];
        si.t = t;
        const TileSpan sp = tile_span(t, tile);
        const uint64_t b0 = sp.b0;
        const uint32_t nb = sp.nb, phase = sp.phase, bytes = sp.bytes;
        const uint8_t* src = sp.src;
        if (t.fmt == KF_FP8_ROW_BF16 || t.fmt == KF_FP8_ROW_FP16) {  // one division per tile
            const uint64_t e0 = b0 * 16u;
            si.row0 = e0 / t.blocks_per_div;
            si.col0 = e0 - si.row0 * t.blocks_per_div;
        }
        si.block0 = b0;
        si.nb = nb;
        si.phase = phase;
        uint32_t nv_tab = 0;
        if (t.fmt == KF_NVFP4 && H.tab_valid) {
            const uint64_t d0 = b0 / t.blocks_per_div, d1 = (b0 + nb - 1u) / t.blocks_per_div;
            if (d0 != nv_d || di != nv_di) {
                nv_same = __float_as_uint(load_f32_bytes(t.divs + 4u * d0)) == H.tab_bits;
                nv_d = d0;
                nv_di = di;
            }
            nv_tab = d0 == d1 && nv_same;
        }
        si.nv_tab = nv_tab;
        mbar_arrive_expect_tx(&H.full[s], bytes);
        bulk_load(inbuf + s * kInStride, src - phase, bytes, &H.full[s]);
    }
    if (fault) atomicOr(p.fault, 1u);
    if (fault || withheld >= 0) {
        // The consumers may have stopped early: wait (bounded) for every copy
        // still in flight before the CTA can exit.  Only the last NST
        // stagings can be in flight (an older stage was reused only after the
        // consumers released it); a withheld staging has no copy.
        for (int j = issued - NST; j < issued; ++j)
            if (j >= 0 && j != withheld)
                mbar_wait_bounded(&H.full[j % NST], static_cast<uint32_t>((j / NST) & 1));
    }
}

// FSEL / OSEL: the launch's format and output type when every tensor shares
// them (the host picks the instantiation), else -1; FSEL == kFselKQuantMix
// for a launch whose tensors are all gguf:q8_0, gguf:q4_k or gguf:q6_k.
template <int FSEL, int OSEL>
__global__ void __launch_bounds__(kBlockThreads, 2) k_decode(const KParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr bool kStaged = decode_staged(FSEL, OSEL);
    constexpr int NST = decode_stages(FSEL);
    uint8_t* inbuf = smem;
    SmemHdr& H = *reinterpret_cast<SmemHdr*>(smem + NST * kInStride);
    uint8_t* outbuf = smem + NST * kInStride + kHdrBytes;  // (16-bit outputs only)
    float* tab = reinterpret_cast<float*>(outbuf + (kStaged ? kOutStageBytes : 0));
    const uint32_t tid = threadIdx.x;
    constexpr bool kLut = uses_lut16(FSEL, OSEL);

    // Shared-memory set-up that reads nothing another kernel writes runs
    // before the wait below, overlapping the previous kernel's tail.
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&H.full[s], 1);
            mbar_init(&H.empty[s], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < 16) {
        H.lut_iq4[tid] = static_cast<float>(c_iq4[tid]);
        H.lut_v[tid] = static_cast<float>(c_v[tid]);
    }

    // A single-tensor launch knows its tiles from its parameters: the
    // producer warms L2 with this CTA's first spans while the previous
    // kernel of the stream may still run.  A prefetch returns no data to the
    // CTA, so it cannot observe that kernel's unfinished writes (L2 is where
    // they land); the staging copies read the spans after the wait below.
    if (p.table == nullptr && tid == kThreads) {
        for (int j = 0; j < NST; ++j) {
            const uint64_t tile = blockIdx.x + static_cast<uint64_t>(j) * gridDim.x;
            if (tile >= p.total_tiles) break;
            const TileSpan sp = tile_span(p.single, tile);
            prefetch_l2(sp.src - sp.phase, sp.bytes);
        }
    }

    // Programmatic dependent launch: this grid may have started before the
    // previous kernel of the stream finished; wait for it (and the
    // visibility of its writes) before touching global memory, then let the
    // next launch start placing its CTAs as this grid's CTAs finish.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // nvfp4: the tables are built for the first divisor of the first nvfp4
    // tensor of the launch; tiles with another divisor divide per element.
    float dw = 0.0f;
    if (p.nv_index >= 0) dw = load_f32_bytes((p.table ? p.table[p.nv_index] : p.single).divs);
    if (tid == 0) {
        H.tab_bits = __float_as_uint(dw);
        H.tab_valid = p.nv_index >= 0;
    }
    __syncthreads();

    if (tid >= kThreads) {  // producer warp: starts staging while the consumers build the tables
        if (tid == kThreads) producer<NST>(p, H, inbuf);
        return;
    }

    // Consumer warps only from here; they meet at named barrier 1.
    if constexpr (kLut) {
        build_lut16<OSEL>(reinterpret_cast<uint32_t*>(tab), dw, tid, kThreads);
    } else if (p.nv_index >= 0) {
        // Entry 16*s + c is e2m1(c) * e4m3fn(s) / d_w; only codes 0..7
        // divide: the entry of c | 8 is the same quotient with the sign bit
        // flipped (RNE division is odd-symmetric, and (-0)*s/d_w is the
        // negated (+0)*s/d_w).
        for (uint32_t i = tid; i < kTabEntries / 2; i += kThreads) {
            const uint32_t sb = i >> 3, c = i & 7u;
            const float q = __fdiv_rn(__fmul_rn(e2m1(c), e4m3fn(sb)), dw);
            tab[16u * sb + c] = q;
            tab[16u * sb + c + 8u] = __uint_as_float(__float_as_uint(q) ^ 0x80000000u);
        }
        if (tid < 256) {  // per-scale quotients for m = 1 and m = 1.5 (1.5*s is exact)
            const float sc = e4m3fn(tid);
            H.nv_q[tid] = make_float2(__fdiv_rn(sc, dw), __fdiv_rn(__fmul_rn(1.5f, sc), dw));
        }
        if (tid < 16) {  // E2M1 code c = 2^k * m: selector of Q_m and +-2^k (+-0 for zero codes)
            const uint32_t e = (tid >> 1) & 3u, m = tid & 1u;
            const bool half = (e >= 1u) && m;  // magnitudes 1.5, 3, 6
            const float scale = (e == 0u) ? (m ? 0.5f : 0.0f) : __uint_as_float((e + 126u) << 23);
            H.nv_code[tid] = make_uint2(half ? 0x7654u : 0x3210u,
                                        __float_as_uint(scale) | ((tid & 8u) ? 0x80000000u : 0u));
        }
        if (tid < 8) H.nv_ok[tid] = 0u;
        asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
        // verify the per-scale form against the table, scale byte by scale byte
        for (uint32_t sb = tid; sb < 256u; sb += kThreads) {
            const float2 q = H.nv_q[sb];
            bool ok = true;
            for (uint32_t c = 0; c < 16u; ++c) {
                const uint2 k = H.nv_code[c];
                const float v = __fmul_rn(__uint_as_float(__byte_perm(__float_as_uint(q.x), __float_as_uint(q.y), k.x)),
                                          __uint_as_float(k.y));
                const float w = tab[16u * sb + c];
                ok = ok && ((w != w) ? (v != v) : (__float_as_uint(v) == __float_as_uint(w)));
            }
            if (ok) atomicOr(&H.nv_ok[sb >> 5], 1u << (sb & 31u));
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");

    // consumer warps
    const uint64_t grid = gridDim.x;
    const uint32_t lane = tid & 31u, warp = tid >> 5;
    uint8_t* const wbuf = outbuf + warp * (2u * kOutBufBytes);  // this warp's two output buffers
    uint32_t nstore = 0;  // bulk copies this warp issued (lane 0); buffer nstore & 1 is the next one
    int it = 0;
    for (uint64_t tile = blockIdx.x; tile < p.total_tiles; tile += grid, ++it) {
        const int s = it % NST;
        // (decided by the whole warp: the decoders shuffle between lanes)
        if (!__all_sync(0xffffffffu,
                        mbar_wait_bounded(&H.full[s], static_cast<uint32_t>((it / NST) & 1), p.wait_ns))) {
            if (lane == 0) {
                atomicOr(p.fault, 2u);
                if (kStaged) bulk_wait_all();  // (the output buffers stay until their copies are read)
            }
            return;
        }
        const StageInfo& si = H.info[s];
        const uint8_t* in = inbuf + s * kInStride;
        const bool nv = (FSEL < 0 || FSEL == KF_NVFP4) && si.t.fmt == KF_NVFP4;
        if (si.phase != 0u || (nv && !si.nv_tab)) {
            // (the byte-table kernels hold no quotient table: nvfp4 divides)
            const Ctx xs{&H, (!kLut && si.nv_tab) ? tab : nullptr, si.t.divs, si.block0, si.t.blocks_per_div,
                         p.grids, code_count(si.t), si.row0, si.col0};
            if (FSEL >= 0)
                decode_tile_slow_one<(FSEL >= 0 ? FSEL : 0), OSEL>(si, in, xs, tid);
            else
                decode_tile_slow(si, in, xs, tid);
        } else {
            const Ctx xf{&H, tab, si.t.divs, si.block0, si.t.blocks_per_div, p.grids, code_count(si.t), si.row0,
                         si.col0};
            if constexpr (kStaged) {
                // A full tile to a 16-byte-aligned 16-bit output: each warp
                // decodes its 1024 outputs into its own buffer and copies them
                // to y with one bulk copy (whole lines, no per-lane stores).
                const bool out16 = OSEL >= 0 || si.t.out == KO_F16 || si.t.out == KO_BF16;
                const bool kq = FSEL != kFselKQuantMix || si.t.fmt == KF_Q8_0 || si.t.fmt == KF_Q4_K ||
                                si.t.fmt == KF_Q6_K;
                const bool full = si.nb == si.t.bpt &&
                                  (!is_fp8_row(si.t.fmt) || (si.block0 + si.nb) * 16u <= code_count(si.t));
                if (out16 && kq && full && si.t.yvec) {
                    uint8_t* ob = wbuf + (nstore & 1u) * kOutBufBytes;
                    if (lane == 0) bulk_wait_read<1>();  // this buffer's previous copy has read it
                    __syncwarp();
                    decode_warp16_fast<FSEL, OSEL>(si, in, xf, reinterpret_cast<const uint4*>(tab), warp, lane, ob);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        // (the destination comes from the stage header, which
                        // the producer rewrites once the stage is released)
                        uint16_t* y = static_cast<uint16_t*>(si.t.y) + si.block0 * si.t.B + warp * kWarpOut;
                        mbar_arrive(&H.empty[s]);
                        bulk_store(y, ob, kOutBufBytes);
                        bulk_commit();
                    }
                    ++nstore;
                    continue;
                }
            }
            if constexpr (kLut) {
                decode_tile_lut16(si, in, reinterpret_cast<const uint4*>(tab), tid);
            } else {
                decode_tile_fast<FSEL, OSEL>(si, in, xf, tid);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&H.empty[s]);
    }
    if (kStaged && lane == 0) bulk_wait_all();
}

// Kernel of format F for output type `osel` (launches that mix output types
// use the generic kernel, so there is no per-format one for them).
template <int F>
KernelFn kernel_row(int osel) {
    switch (osel) {
        case KO_F32: return k_decode<F, KO_F32>;
        case KO_F16: return k_decode<F, KO_F16>;
        case KO_BF16: return k_decode<F, KO_BF16>;
        case KO_F64: return k_decode<F, KO_F64>;
        default: return nullptr;
    }
}

}  // namespace
}  // namespace ndq
