// ndq_matvec.cuh -- decode fused into a matrix product with few activation
// rows (matrix-vector shaped work: token-by-token generation).
//
//     Y[m, n] = sum_k X[m, k] * W[n, k],   m < M <= kMvMaxRows, n < N
//
// W is the payload decoded exactly as DequantizePacked does (binary32), or
// that decode rounded once to bfloat16 (the weight operand a decode-to-bf16
// + bf16 product would use); X is bfloat16 [M, K]; products and sums are
// binary32 FMAs (NInfer "tensor-formats": a consuming kernel chooses its own
// fusion, reduction order and intermediate precision).  The result is
// deterministic: every output is summed in a fixed order.
//
// Four kernels: k_gemvl (one row of X, the formats of a K-quant model,
// lean per-format decoders and X in registers; below), k_gemvm (1 to 8 rows
// of X, the same decoders, X in shared memory; below), k_gemv1 (one row of
// X, any format; below) and k_matvec (up to 8 rows of X).  k_matvec's CTA
// layout is the decode kernel's: one producer warp stages payload units
// into the shared-memory ring with bulk copies; 8 consumer warps decode
// 16-element chunks with the same Fmt<F> decoders and accumulate against X.
// A unit is R = rows_per_stage whole weight rows (K <= 8192/R),
// or, when K > 4096, a segment of up to 8192 elements of one row.  Each CTA
// owns whole units, so a row's partial sums meet in the CTA: the 256/R
// threads of a row group take its chunks in turn; warp shuffles, then one
// partial per warp in shared memory; the last warp of the group to finish
// adds the group's partials in warp order and writes Y.
#pragma once

#include "ndq_device.cuh"
#include "ndq_fused.h"

namespace ndq {
namespace {

struct MvStage {
    uint64_t row;     // first weight row of the unit
    uint64_t k0;      // first column of the unit (a segment's offset; 0 for whole rows)
    uint64_t block0;  // first block of the unit in the payload
    uint32_t nb;      // blocks per row in the unit (the segment's, or the row's)
    uint32_t phase;   // byte offset of the first block within the stage
    uint32_t last;    // 1 when the unit ends its rows
    uint32_t nrows;   // rows in the unit (1 for a segment)
    uint32_t pad[2];
};
static_assert(sizeof(MvStage) == 48, "MvStage layout");

struct MvShared {
    MvStage st[kStages];
    float red[kStages][kConsumerWarps][kMvMaxRows];  // per-warp partial sums of a row
    uint32_t done[kStages][kConsumerWarps];          // per row group: warps that stored their partials
};

constexpr int kMvExtraBytes = (sizeof(MvShared) + 127) / 128 * 128;

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Accumulate this thread's chunks of one staged unit into acc: the thread's
// row group g = tid / (256/R) owns row g of the unit, whose nb blocks hold
// nb*CPB chunks; the group's threads take them in turn.  Products and sums
// are binary32 fused multiply-adds, two lanes at a time (even and odd
// elements of a chunk in the two lanes of a pair).  XM says where the
// activations come from: kMvXF32, one row converted to binary32 in shared
// memory (acc[0..1], four chains); kMvXBf16, the launch's rows as bfloat16 in
// shared memory; kMvXGlobal, bfloat16 from global memory (acc[m] per row).
template <int F, bool PH, int MT, int XM>
__device__ __forceinline__ void mv_tile(const MvStage& st, const uint8_t* in, const Ctx& x, uint32_t tid,
                                        const MvParams& p, const uint8_t* xs, float2* acc) {
    using Fm = Fmt<F>;
    constexpr int CE = Fm::CE;
    const uint32_t gsize = kThreads / static_cast<uint32_t>(p.rows_per_stage);
    const uint32_t g = tid / gsize;
    if (g >= st.nrows) return;
    const uint32_t per_row = st.nb * static_cast<uint32_t>(Fm::CPB);
    const uint32_t ph = PH ? st.phase : 0u;
    for (uint32_t j = tid - g * gsize; j < per_row; j += gsize) {
        const uint32_t c = g * per_row + j;
        float v[CE];
        Fm::template chunk<PH>(in, ph, c, v, x);
        if (p.wbf16) {  // round the decoded weights once to bfloat16
#pragma unroll
            for (int i = 0; i < CE / 2; ++i) {
                const uint32_t u = pack_bf16(v[2 * i], v[2 * i + 1]);
                v[2 * i] = bf16_lo(u);
                v[2 * i + 1] = bf16_hi(u);
            }
        }
        const uint64_t col = st.k0 + static_cast<uint64_t>(CE) * j;  // column of the chunk's first weight
        // (shared-memory copies: piece q of chunk jj of row m at piece index
        // (m * CE/w + q) * K/CE + jj, so that the lanes' consecutive chunks
        // are consecutive 16-byte pieces, free of bank conflicts)
        const uint64_t nj = p.K / static_cast<uint64_t>(CE), jj = col / static_cast<uint64_t>(CE);
        if constexpr (XM == kMvXF32) {
#pragma unroll
            for (int q = 0; q < CE / 4; ++q) {
                const float4 xv = reinterpret_cast<const float4*>(xs)[static_cast<uint64_t>(q) * nj + jj];
                acc[0] = fma2(make_float2(xv.x, xv.y), make_float2(v[4 * q], v[4 * q + 1]), acc[0]);
                acc[1] = fma2(make_float2(xv.z, xv.w), make_float2(v[4 * q + 2], v[4 * q + 3]), acc[1]);
            }
        } else {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (MT == 1 || m < p.m) {
                    uint32_t xb[CE / 2];
                    if (XM == kMvXBf16) {
#pragma unroll
                        for (int q = 0; q < CE / 8; ++q) {
                            const uint4 t =
                                reinterpret_cast<const uint4*>(xs)[(static_cast<uint64_t>(m) * (CE / 8) + q) * nj + jj];
                            xb[4 * q] = t.x;
                            xb[4 * q + 1] = t.y;
                            xb[4 * q + 2] = t.z;
                            xb[4 * q + 3] = t.w;
                        }
                    } else {
                        const uint16_t* xr = p.x + static_cast<uint64_t>(m) * p.K + col;
                        if (p.xvec) {
#pragma unroll
                            for (int q = 0; q < CE / 8; ++q) {
                                const uint4 t = __ldg(reinterpret_cast<const uint4*>(xr) + q);
                                xb[4 * q] = t.x;
                                xb[4 * q + 1] = t.y;
                                xb[4 * q + 2] = t.z;
                                xb[4 * q + 3] = t.w;
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < CE / 2; ++i)
                                xb[i] = static_cast<uint32_t>(__ldg(xr + 2 * i)) |
                                        (static_cast<uint32_t>(__ldg(xr + 2 * i + 1)) << 16);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < CE / 2; ++i)
                        acc[m] = fma2(make_float2(bf16_lo(xb[i]), bf16_hi(xb[i])), make_float2(v[2 * i], v[2 * i + 1]),
                                      acc[m]);
                }
            }
        }
    }
}

// Payload span of unit u's sb-th segment (rows are whole when R > 1).
struct MvSpan {
    const uint8_t* src;
    uint32_t nrows, nb, phase, bytes;
};
__device__ __forceinline__ MvSpan mv_span(const MvParams& p, uint64_t u, uint64_t sb, uint64_t seg) {
    const DevTensor& t = p.w;
    const uint64_t R = static_cast<uint64_t>(p.rows_per_stage);
    const uint64_t row0 = u * R;
    MvSpan r;
    r.nrows = static_cast<uint32_t>(p.n_rows - row0 < R ? p.n_rows - row0 : R);
    const uint64_t left = p.bpr - sb;
    r.nb = static_cast<uint32_t>(left < seg ? left : seg);
    r.src = t.x + (row0 * p.bpr + sb) * t.S;
    r.phase = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(r.src) & 15u);
    r.bytes = (r.phase + r.nrows * r.nb * t.S + 15u) & ~15u;
    return r;
}

// Units in the order both the producer and the consumers walk them: unit
// u = blockIdx.x + i*gridDim.x covers rows [u*R, u*R + R) (whole rows), or
// row u when rows are segmented (R == 1), then its segments in order.
__device__ void mv_producer(const MvParams& p, SmemHdr& H, MvShared& S, uint8_t* inbuf) {
    const DevTensor& t = p.w;
    const uint64_t R = static_cast<uint64_t>(p.rows_per_stage);
    const uint64_t seg = R > 1 ? p.bpr : static_cast<uint64_t>(t.bpt);  // blocks per row per unit
    const uint64_t units = (p.n_rows + R - 1) / R;
    int issued = 0;
    bool fault = false;
    for (uint64_t u = blockIdx.x; u < units && !fault; u += gridDim.x) {
        const uint64_t row0 = u * R;
        const uint32_t nrows = static_cast<uint32_t>(p.n_rows - row0 < R ? p.n_rows - row0 : R);
        for (uint64_t sb = 0; sb < p.bpr; sb += seg, ++issued) {
            const int s = issued % kStages;
            if (issued >= kStages &&
                !mbar_wait_bounded(&H.empty[s], static_cast<uint32_t>(((issued / kStages) - 1) & 1))) {
                fault = true;
                break;
            }
            const MvSpan sp = mv_span(p, u, sb, seg);
            const uint32_t nb = sp.nb, phase = sp.phase, bytes = sp.bytes;
            const uint64_t b0 = row0 * p.bpr + sb;
            const uint8_t* src = sp.src;
            MvStage& st = S.st[s];
            st.row = row0;
            st.k0 = sb * t.B;
            st.block0 = b0;
            st.nb = nb;
            st.phase = phase;
            st.last = (sb + seg >= p.bpr) ? 1u : 0u;
            st.nrows = nrows;
            mbar_arrive_expect_tx(&H.full[s], bytes);
            bulk_load(inbuf + s * kInStride, src - phase, bytes, &H.full[s]);
        }
    }
    if (fault) {
        atomicOr(p.fault, 1u);
        for (int j = issued - kStages; j < issued; ++j)
            if (j >= 0) mbar_wait_bounded(&H.full[j % kStages], static_cast<uint32_t>((j / kStages) & 1));
    }
}

// Kernels of decode family F; the output type is a launch parameter (it
// only changes the final store).  MT: activation rows per launch at most (1
// or kMvMaxRows).  ALIGNED: every staged unit starts on a 16-byte boundary
// (a 16-byte-aligned payload whose row groups span whole 16-byte lines), so
// the decoders read at byte phase 0; otherwise they take the phase-tolerant
// loads.  XM: where the activations are read (see mv_tile); the shared-memory
// copies follow the CTA's other shared memory.
template <int F, int MT, bool ALIGNED, int XM>
__global__ void __launch_bounds__(kBlockThreads, 2) k_matvec(const MvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* inbuf = smem;
    SmemHdr& H = *reinterpret_cast<SmemHdr*>(smem + kStages * kInStride);
    MvShared& S = *reinterpret_cast<MvShared*>(smem + kStages * kInStride + kHdrBytes);
    uint8_t* xs = smem + kStages * kInStride + kHdrBytes + kMvExtraBytes;
    const uint32_t tid = threadIdx.x;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&H.full[s], 1);
            mbar_init(&H.empty[s], kConsumerWarps);
            for (int g = 0; g < kConsumerWarps; ++g) S.done[s][g] = 0u;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        H.tab_valid = 0;
    }
    if (tid < 16) {
        H.lut_iq4[tid] = static_cast<float>(c_iq4[tid]);
        H.lut_v[tid] = static_cast<float>(c_v[tid]);
    }
    const uint64_t R = static_cast<uint64_t>(p.rows_per_stage);
    const uint64_t seg = R > 1 ? p.bpr : static_cast<uint64_t>(p.w.bpt);  // blocks per row per unit
    // The weights are the launch's parameters: warm L2 with this CTA's first
    // spans while the previous kernel of the stream may still run (a
    // prefetch returns no data to the CTA, so it cannot observe that
    // kernel's unfinished writes; the staging copies read after the wait).
    if (tid == kThreads) {
        const uint64_t units = (p.n_rows + R - 1) / R;
        int n = 0;
        for (uint64_t u = blockIdx.x; u < units && n < kStages; u += gridDim.x)
            for (uint64_t sb = 0; sb < p.bpr && n < kStages; sb += seg, ++n) {
                const MvSpan sp = mv_span(p, u, sb, seg);
                prefetch_l2(sp.src - sp.phase, sp.bytes);
            }
    }
    // Programmatic dependent launch: wait for the previous kernel (it may
    // have written X) before reading global memory, then let the next launch
    // place its CTAs as this grid's CTAs finish.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    if (tid >= kThreads) {  // producer warp
        if (tid == kThreads) mv_producer(p, H, S, inbuf);
        return;
    }

    // The activations into shared memory (binary32 for one row, bfloat16 for
    // several), by the consumer threads, while the producer stages weights;
    // laid out in 16-byte pieces as mv_tile reads them (K is a multiple of
    // the chunk width CE here).
    constexpr int CE = Fmt<F>::CE;
    if constexpr (XM == kMvXF32) {
        const uint64_t nj = p.K / CE, npc = nj * (CE / 4);  // pieces of 4 values
        float4* x4 = reinterpret_cast<float4*>(xs);
        for (uint64_t i = tid; i < npc; i += kThreads) {  // piece i = q * nj + jj
            const uint64_t q = i / nj, jj = i - q * nj, e = jj * CE + 4u * q;
            uint32_t a, b;
            if (p.xvec) {
                const uint2 t = __ldg(reinterpret_cast<const uint2*>(p.x + e));
                a = t.x;
                b = t.y;
            } else {
                a = static_cast<uint32_t>(__ldg(p.x + e)) | (static_cast<uint32_t>(__ldg(p.x + e + 1)) << 16);
                b = static_cast<uint32_t>(__ldg(p.x + e + 2)) | (static_cast<uint32_t>(__ldg(p.x + e + 3)) << 16);
            }
            x4[i] = make_float4(bf16_lo(a), bf16_hi(a), bf16_lo(b), bf16_hi(b));
        }
    } else if constexpr (XM == kMvXBf16) {  // (K % 8 == 0 and X 16-byte aligned)
        const uint64_t nj = p.K / CE, per = nj * (CE / 8), n16 = static_cast<uint64_t>(p.m) * per;
        for (uint64_t i = tid; i < n16; i += kThreads) {  // piece i = (m * CE/8 + q) * nj + jj
            const uint64_t m = i / per, r = i - m * per, q = r / nj, jj = r - q * nj;
            reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(p.x + m * p.K + jj * CE + 8u * q));
        }
    }
    if constexpr (XM != kMvXGlobal) asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");

    const uint32_t lane = tid & 31u, warp = tid >> 5;
    const DevTensor& t = p.w;
    const Ctx base{&H, nullptr, t.divs, 0, t.blocks_per_div, p.grids, code_count(t), 0, 0};
    const uint64_t units = (p.n_rows + R - 1) / R;
    const uint32_t gwarps = static_cast<uint32_t>(kConsumerWarps / R);  // warps per row group
    const uint32_t g = warp / gwarps;                                    // this warp's row group
    constexpr int NA = (XM == kMvXF32) ? 2 : MT;                         // pair accumulators
    float2 acc[NA];
#pragma unroll
    for (int m = 0; m < NA; ++m) acc[m] = make_float2(0.0f, 0.0f);
    int it = 0;
    for (uint64_t u = blockIdx.x; u < units; u += gridDim.x) {
        for (uint64_t sb = 0; sb < p.bpr; sb += seg, ++it) {
            const int s = it % kStages;
            if (!mbar_wait_bounded(&H.full[s], static_cast<uint32_t>((it / kStages) & 1))) {
                if (lane == 0) atomicOr(p.fault, 2u);
                return;
            }
            const MvStage& st = S.st[s];
            const uint8_t* in = inbuf + s * kInStride;
            Ctx x = base;
            x.block0 = st.block0;
            x.row0 = st.row;  // fp8 rows: the unit's first code is at (row, k0)
            x.col0 = st.k0;
            mv_tile<F, !ALIGNED, MT, XM>(st, in, x, tid, p, xs, acc);
            if (st.last && g < st.nrows) {
                // warp partials, then the last warp of the row group adds the
                // group's partials in warp order
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (MT == 1 || m < p.m) {
                        float v = (XM == kMvXF32) ? __fadd_rn(__fadd_rn(acc[0].x, acc[0].y), __fadd_rn(acc[1].x, acc[1].y))
                                                  : __fadd_rn(acc[m].x, acc[m].y);
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                        if (lane == 0) S.red[s][warp][m] = v;
                    }
                }
#pragma unroll
                for (int m = 0; m < NA; ++m) acc[m] = make_float2(0.0f, 0.0f);
                uint32_t prior = 0;
                if (lane == 0) {
                    __threadfence_block();
                    prior = atomicAdd(&S.done[s][g], 1u);
                }
                prior = __shfl_sync(0xffffffffu, prior, 0);
                if (prior == gwarps - 1) {  // every warp of the group has stored its partial
                    __threadfence_block();
                    if (lane < static_cast<uint32_t>(p.m)) {
                        float sum = 0.0f;
                        for (uint32_t w = g * gwarps; w < (g + 1) * gwarps; ++w)
                            sum = __fadd_rn(sum, *reinterpret_cast<volatile float*>(&S.red[s][w][lane]));
                        const uint64_t o = static_cast<uint64_t>(lane) * p.n_rows + st.row + g;
                        if (p.out_bf16)
                            static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(sum);
                        else
                            static_cast<float*>(p.y)[o] = sum;
                    }
                    __syncwarp();
                    if (lane == 0) S.done[s][g] = 0u;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&H.empty[s]);
        }
    }
}

// ---------------------------------------------------------------------------
// One activation row (token-by-token generation): k_gemv1.  Each consumer
// warp owns one weight row of a block of 8 rows and walks it in segments of
// kGvSeg weights; a stage holds the current segment of all 8 rows (8 bulk
// copies, one per row).  A lane takes every 32nd 16-weight chunk of its
// warp's segment, so a row's partial sums stay in one warp until its last
// segment, where 5 shuffles add them and lane 0 writes the output: no
// exchange between warps.  The activation row sits in shared memory as
// binary32, converted once per CTA, in the bank-conflict-free piece layout of
// mv_tile.
// ---------------------------------------------------------------------------
constexpr int kGvSeg = 2048;                 // weights per row segment
constexpr int kGvStages = 3;
constexpr int kGvRows = kConsumerWarps;      // rows per block: one per warp

// Bytes of one row-segment slot of format F: the segment's blocks, the
// phase of an unaligned start and the decoders' over-read, in 128-byte units.
__host__ __device__ constexpr uint32_t gv_slot_bytes(uint32_t B, uint32_t S) {
    return ((kGvSeg / B) * S + 48u + 127u) / 128u * 128u;
}
template <int F>
__host__ __device__ constexpr uint32_t gv_slot_bytes() {
    return gv_slot_bytes(Fmt<F>::B, Fmt<F>::S);
}
// Dynamic shared memory of k_gemv1 without the activation row (the kernel's
// blocks hold B decoded values in S bytes).
inline size_t gemv1_smem_base(uint32_t B, uint32_t S) {
    return static_cast<size_t>(kGvStages * kGvRows * gv_slot_bytes(B, S) + kHdrBytes + kMvExtraBytes);
}

struct GvStage {
    uint64_t rb;        // row block
    uint32_t b0;        // first block of the segment within each row
    uint32_t nb;        // blocks of the segment
    uint8_t phase[kGvRows];
};

template <int F>
__device__ void gv_producer(const MvParams& p, SmemHdr& H, GvStage* S, uint8_t* inbuf) {
    constexpr uint32_t kSlot = gv_slot_bytes<F>();
    const DevTensor& t = p.w;
    const uint64_t nrb = (p.n_rows + kGvRows - 1) / kGvRows;
    const uint32_t segb = static_cast<uint32_t>(kGvSeg / t.B < p.bpr ? kGvSeg / t.B : p.bpr);
    int issued = 0;
    bool fault = false;
    for (uint64_t rb = blockIdx.x; rb < nrb && !fault; rb += gridDim.x) {
        for (uint64_t b0 = 0; b0 < p.bpr; b0 += segb, ++issued) {
            const int s = issued % kGvStages;
            if (issued >= kGvStages &&
                !mbar_wait_bounded(&H.empty[s], static_cast<uint32_t>(((issued / kGvStages) - 1) & 1))) {
                fault = true;
                break;
            }
            const uint32_t nb = static_cast<uint32_t>(p.bpr - b0 < segb ? p.bpr - b0 : segb);
            GvStage& st = S[s];
            st.rb = rb;
            st.b0 = static_cast<uint32_t>(b0);
            st.nb = nb;
            const uint8_t* src[kGvRows];
            uint32_t bytes[kGvRows], total = 0;
#pragma unroll
            for (int w = 0; w < kGvRows; ++w) {
                const uint64_t row = rb * kGvRows + w;
                bytes[w] = 0;
                src[w] = nullptr;
                if (row < p.n_rows) {
                    const uint8_t* a = t.x + (row * p.bpr + b0) * t.S;
                    const uint32_t ph = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(a) & 15u);
                    st.phase[w] = static_cast<uint8_t>(ph);
                    src[w] = a - ph;
                    bytes[w] = (ph + nb * t.S + 15u) & ~15u;
                    total += bytes[w];
                }
            }
            mbar_arrive_expect_tx(&H.full[s], total);
            uint8_t* dst = inbuf + static_cast<uint32_t>(s) * (kGvRows * kSlot);
#pragma unroll
            for (int w = 0; w < kGvRows; ++w)
                if (bytes[w]) bulk_load(dst + w * kSlot, src[w], bytes[w], &H.full[s]);
        }
    }
    if (fault) {
        atomicOr(p.fault, 1u);
        for (int j = issued - kGvStages; j < issued; ++j)
            if (j >= 0) mbar_wait_bounded(&H.full[j % kGvStages], static_cast<uint32_t>((j / kGvStages) & 1));
    }
}

// Round decoded weights once to bfloat16 when the launch asks for bfloat16
// weights.
template <int N>
__device__ __forceinline__ void gv_round_bf16(const MvParams& p, float* v) {
    if (p.wbf16) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const uint32_t u = pack_bf16(v[2 * i], v[2 * i + 1]);
            v[2 * i] = bf16_lo(u);
            v[2 * i + 1] = bf16_hi(u);
        }
    }
}

// acc += X . W over one chunk: its CE / 4 activation pieces are xr[q * nj].
template <int CE>
__device__ __forceinline__ void gv_fma(const float4* xr, uint32_t nj, const float* v, float2& a0, float2& a1) {
#pragma unroll
    for (int q = 0; q < CE / 4; ++q) {
        const float4 xv = xr[q * nj];
        a0 = fma2(make_float2(xv.x, xv.y), make_float2(v[4 * q], v[4 * q + 1]), a0);
        a1 = fma2(make_float2(xv.z, xv.w), make_float2(v[4 * q + 2], v[4 * q + 3]), a1);
    }
}

// ALIGNED: the payload and every row start are 16-byte aligned (every
// segment then starts at byte phase 0).
template <int F, bool ALIGNED>
__global__ void __launch_bounds__(kBlockThreads, 2) k_gemv1(const MvParams p) {
    using Fm = Fmt<F>;
    constexpr int CE = Fm::CE;
    constexpr uint32_t kSlot = gv_slot_bytes<F>();
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* inbuf = smem;
    constexpr uint32_t kIn = kGvStages * kGvRows * kSlot;
    SmemHdr& H = *reinterpret_cast<SmemHdr*>(smem + kIn);
    GvStage* S = reinterpret_cast<GvStage*>(smem + kIn + kHdrBytes);
    float4* x4 = reinterpret_cast<float4*>(smem + kIn + kHdrBytes + kMvExtraBytes);
    const uint32_t tid = threadIdx.x;

    if (tid == 0) {
        for (int s = 0; s < kGvStages; ++s) {
            mbar_init(&H.full[s], 1);
            mbar_init(&H.empty[s], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < 16) {
        H.lut_iq4[tid] = static_cast<float>(c_iq4[tid]);
        H.lut_v[tid] = static_cast<float>(c_v[tid]);
    }
    const uint64_t nrb = (p.n_rows + kGvRows - 1) / kGvRows;
    // warm L2 with this CTA's first row block (see k_matvec)
    if (tid >= kThreads && blockIdx.x < nrb) {
        const uint32_t w = tid - kThreads;
        const uint64_t row = blockIdx.x * static_cast<uint64_t>(kGvRows) + (w & 7u);
        if (w < kGvRows && row < p.n_rows) {
            const uint8_t* a = p.w.x + row * p.bpr * p.w.S;
            const uint32_t ph = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(a) & 15u);
            const uint64_t rb = (ph + p.bpr * p.w.S + 15u) & ~15ull;
            prefetch_l2(a - ph, static_cast<uint32_t>(rb < 16384u ? rb : 16384u));
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    if (tid >= kThreads) {
        if (tid == kThreads) gv_producer<F>(p, H, S, inbuf);
        return;
    }

    // the activation row as binary32 pieces (piece q * K/CE + jj holds
    // values CE*jj + 4q .. +3)
    const uint64_t nj = p.K / CE;
    {
        const uint64_t npc = nj * (CE / 4);
        for (uint64_t i = tid; i < npc; i += kThreads) {
            const uint64_t q = i / nj, jj = i - q * nj, e = jj * CE + 4u * q;
            uint32_t a, b;
            if (p.xvec) {
                const uint2 t = __ldg(reinterpret_cast<const uint2*>(p.x + e));
                a = t.x;
                b = t.y;
            } else {
                a = static_cast<uint32_t>(__ldg(p.x + e)) | (static_cast<uint32_t>(__ldg(p.x + e + 1)) << 16);
                b = static_cast<uint32_t>(__ldg(p.x + e + 2)) | (static_cast<uint32_t>(__ldg(p.x + e + 3)) << 16);
            }
            x4[i] = make_float4(bf16_lo(a), bf16_hi(a), bf16_lo(b), bf16_hi(b));
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");

    const uint32_t lane = tid & 31u, warp = tid >> 5;
    const DevTensor& t = p.w;
    const uint32_t nj32 = static_cast<uint32_t>(nj);  // (K * 4 <= kMvXBytes)
    const uint32_t segb = static_cast<uint32_t>(kGvSeg / t.B < p.bpr ? kGvSeg / t.B : p.bpr);
    Ctx x{&H, nullptr, t.divs, 0, t.blocks_per_div, p.grids, code_count(t), 0, 0};
    float2 a0 = make_float2(0.0f, 0.0f), a1 = make_float2(0.0f, 0.0f);
    int it = 0;
    for (uint64_t rb = blockIdx.x; rb < nrb; rb += gridDim.x) {
        const uint64_t row = rb * kGvRows + warp;
        for (uint64_t b0 = 0; b0 < p.bpr; b0 += segb, ++it) {
            const int s = it % kGvStages;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&H.full[s], static_cast<uint32_t>((it / kGvStages) & 1)))) {
                if (lane == 0) atomicOr(p.fault, 2u);
                return;
            }
            if (row < p.n_rows) {
                const GvStage& st = S[s];
                const uint8_t* in = inbuf + static_cast<uint32_t>(s) * (kGvRows * kSlot) + warp * kSlot;
                const uint32_t ph = ALIGNED ? 0u : st.phase[warp];
                x.block0 = row * p.bpr + b0;
                x.row0 = row;
                x.col0 = b0 * t.B;
                const uint32_t nch = st.nb * static_cast<uint32_t>(Fm::CPB);
                const float4* xr0 = x4 + b0 * t.B / CE;  // this segment's first piece
                for (uint32_t c = lane; c < nch; c += 32u) {
                    float v[CE];
                    Fm::template chunk<!ALIGNED>(in, ph, c, v, x);
                    gv_round_bf16<CE>(p, v);
                    gv_fma<CE>(xr0 + c, nj32, v, a0, a1);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&H.empty[s]);
        }
        if (row < p.n_rows) {  // the row's sum: its lanes' chains, then the warp
            float v = __fadd_rn(__fadd_rn(a0.x, a0.y), __fadd_rn(a1.x, a1.y));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) {
                if (p.out_bf16)
                    static_cast<__nv_bfloat16*>(p.y)[row] = __float2bfloat16_rn(v);
                else
                    static_cast<float*>(p.y)[row] = v;
            }
        }
        a0 = make_float2(0.0f, 0.0f);
        a1 = make_float2(0.0f, 0.0f);
    }
}

// ---------------------------------------------------------------------------
// One activation row, lean decoders: k_gemvl.  For the formats of a K-quant
// model (gguf q8_0, q4_k, q6_k) with K a multiple of 512 and 16-byte-aligned
// rows, of one tensor or of up to 8 tensors that share X (one launch for,
// say, the q, k and v projections).  A stage holds rb consecutive whole
// weight rows of one tensor (one bulk copy); the CTAs take row blocks in
// turn.  A row is cut into lane units of 16 weights,
// 32 per warp iteration; warp w always takes the same XR iterations of every
// row, so its lanes keep their activations in registers (binary32, loaded
// once per CTA) and reuse them for the stage's rb rows, whose sums are
// independent chains.  A unit is the 16 weights that a lane decodes from a
// few aligned 32-bit words of one block (for q6_k, 4 runs of 4 from two
// low-nibble words and one high-bit word), so the decoders do no per-chunk
// realignment; the lanes of a group of four share their block's scales by
// shuffles.  A warp reduces its rb row sums together (a reduce-scatter over
// the lanes, then a butterfly) and stores one partial per row; the last warp
// of the stage adds each row's partials in warp order and writes y.
// Products and sums are binary32 (FMA pairs); W is the exact decode (or its
// bfloat16 rounding), formed exactly as the decode kernels do.
// ---------------------------------------------------------------------------
constexpr int kGlStages = 3;
constexpr uint32_t kGlIter = 512;     // weights per warp iteration (32 lanes x 16)
constexpr uint32_t kGlMaxRows = 8;    // rows per stage
constexpr uint32_t kGlSlotMax = 36u * 1024u;

// Bytes of one stage slot of rb rows: the rows and the decoders' over-read
// (at most 4 bytes past the last row's last byte), in 128-byte units.
__host__ __device__ constexpr uint32_t gl_slot_bytes(uint64_t row_bytes, uint32_t rb) {
    return static_cast<uint32_t>((row_bytes * rb + 16u + 127u) / 128u * 128u);
}

struct GlShared {
    float red[kGlStages][kGlMaxRows][kConsumerWarps];  // per-warp partial sums of the staged rows
    uint32_t cnt[kGlStages];                           // warps that stored their partials
};

inline size_t gemvl_smem_bytes(uint32_t slot) {
    return static_cast<size_t>(kGlStages) * slot + kHdrBytes + (sizeof(GlShared) + 127u) / 128u * 128u;
}

// Rows per stage for a launch: the most (up to 8, and 2 when a lane holds 4
// units) whose slot fits kGlSlotMax while leaving at least two row blocks per
// resident CTA.
inline uint32_t gemvl_rows_per_stage(uint64_t n_rows, uint64_t row_bytes, uint32_t xr, uint64_t resident) {
    uint32_t rb = xr >= 4u ? 2u : kGlMaxRows;
    while (rb > 1u && (gl_slot_bytes(row_bytes, rb) > kGlSlotMax || (n_rows + rb - 1u) / rb < 2u * resident))
        rb >>= 1;
    return rb;
}

template <bool WBF16>
__device__ __forceinline__ float2 gl_round(float2 v) {
    if (!WBF16) return v;
    const uint32_t u = pack_bf16(v.x, v.y);
    return make_float2(bf16_lo(u), bf16_hi(u));
}

// acc += x[0..3] * (the 4 bytes of w minus the code offset, times d), as
// two FMA pairs.
template <bool WBF16>
__device__ __forceinline__ void gl_mul_acc(float d, uint32_t w, float bias, const float* x, float2& acc) {
    const float2 dd = make_float2(d, d);
    const float2 p = gl_round<WBF16>(mul2(dd, bytes_minus2<0>(w, bias)));
    const float2 q = gl_round<WBF16>(mul2(dd, bytes_minus2<2>(w, bias)));
    acc = fma2(make_float2(x[0], x[1]), p, acc);
    acc = fma2(make_float2(x[2], x[3]), q, acc);
}

// acc += x[0..3] * fma(a, the 4 bytes of w minus the offset, c) (only where
// a times the code is exact, so the FMA rounds the rule's difference once).
template <bool WBF16>
__device__ __forceinline__ void gl_fma_acc(float a, uint32_t w, float bias, float c, const float* x, float2& acc) {
    const float2 aa = make_float2(a, a), cc = make_float2(c, c);
    const float2 p = gl_round<WBF16>(fma2(aa, bytes_minus2<0>(w, bias), cc));
    const float2 q = gl_round<WBF16>(fma2(aa, bytes_minus2<2>(w, bias), cc));
    acc = fma2(make_float2(x[0], x[1]), p, acc);
    acc = fma2(make_float2(x[2], x[3]), q, acc);
}

// The aligned 32-bit word holding bytes [off, off + 4) of the stage, for an
// offset that is a multiple of 2 (two loads and a funnel shift).
__device__ __forceinline__ uint32_t lds_4h(const uint8_t* base, uint32_t off) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(base + (off & ~3u));
    return __funnelshift_r(w[0], w[1], (off & 2u) * 8u);
}

// Pair operations through the compiler's float2 builtins (the same
// correctly rounded lane results as sub2 / mul2 / fma2, which the compiler
// can schedule and place in register pairs itself): used by k_gemvm's
// decoders and products.
__device__ __forceinline__ float2 gm_fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 gm_mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
// Bytes I and I+1 of w as the floats 2^23 + byte, minus `bias` (adding
// -bias rounds as subtracting bias does; both are exact here).
template <int I>
__device__ __forceinline__ float2 gm_bytes_minus2(uint32_t w, float bias) {
    return __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | I)),
                                  __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | (I + 1)))),
                      make_float2(-bias, -bias));
}

template <int F>
struct Gl {
    static constexpr bool kLean = false;
};

// gguf:q8_0: unit u = elements 16u .. 16u + 15 (half u & 1 of block u >> 1).
template <>
struct Gl<KF_Q8_0> {
    static constexpr bool kLean = true;
    __device__ __forceinline__ static uint32_t col(uint32_t u, int r) { return 16u * u + 4u * r; }
    template <bool WBF16>
    __device__ __forceinline__ static void unit(const uint8_t* in, uint32_t u, uint32_t, const float* x,
                                                float2& acc) {
        const uint32_t off = (u >> 1) * 34u;
        const float d = h2f(*reinterpret_cast<const uint16_t*>(in + off));
        const uint4 q = lds_16<false>(in, off + 2u + 16u * (u & 1u));
        const float bias = 8388736.0f;  // 2^23 + 128; XOR 0x80 maps signed to offset-128
        gl_mul_acc<WBF16>(d, q.x ^ 0x80808080u, bias, x, acc);
        gl_mul_acc<WBF16>(d, q.y ^ 0x80808080u, bias, x + 4, acc);
        gl_mul_acc<WBF16>(d, q.z ^ 0x80808080u, bias, x + 8, acc);
        gl_mul_acc<WBF16>(d, q.w ^ 0x80808080u, bias, x + 12, acc);
    }
    // The same unit in two steps for k_gemvm: its fields (prep), then the 4
    // weights of run r (run), bit-identical to unit()'s.
    struct U {
        float d;
        uint4 q;
    };
    __device__ __forceinline__ static U prep(const uint8_t* in, uint32_t u, uint32_t) {
        const uint32_t off = (u >> 1) * 34u;
        U s;
        s.d = h2f(*reinterpret_cast<const uint16_t*>(in + off));
        s.q = lds_16<false>(in, off + 2u + 16u * (u & 1u));
        return s;
    }
    template <bool WBF16>
    __device__ __forceinline__ static void run(const U& s, int r, float2& w01, float2& w23) {
        const uint32_t q = (r == 0 ? s.q.x : r == 1 ? s.q.y : r == 2 ? s.q.z : s.q.w) ^ 0x80808080u;
        const float2 dd = make_float2(s.d, s.d);
        const float bias = 8388736.0f;
        w01 = gl_round<WBF16>(gm_mul2(dd, gm_bytes_minus2<0>(q, bias)));
        w23 = gl_round<WBF16>(gm_mul2(dd, gm_bytes_minus2<2>(q, bias)));
    }
};

// gguf:q4_k: unit u = 16 b + s of block b: i = s >> 2 picks sub-blocks 2i
// (low nibbles) and 2i + 1 (high nibbles) of code bytes 32i .. 32i + 31,
// t = s & 3 the words at 4t and 4t + 16; run r holds elements
// 64i + 4t + 16 (r & 1) + 32 (r >> 1) .. +3.
template <>
struct Gl<KF_Q4_K> {
    static constexpr bool kLean = true;
    __device__ __forceinline__ static uint32_t col(uint32_t u, int r) {
        const uint32_t s = u & 15u;
        return 256u * (u >> 4) + 64u * (s >> 2) + 4u * (s & 3u) + 16u * (r & 1) + 32u * (r >> 1);
    }
    template <bool WBF16>
    __device__ __forceinline__ static void unit(const uint8_t* in, uint32_t u, uint32_t lane, const float* x,
                                                float2& acc) {
        const uint32_t s = u & 15u, i = s >> 2, t = s & 3u;
        const uint8_t* b = in + (u >> 4) * 144u;
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(b + 16u + 32u * i + 4u * t);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(b + 32u + 32u * i + 4u * t);
        // Lane t of the group forms one of M(d, a[2i]), -M(dmin, m[2i]),
        // M(d, a[2i+1]), -M(dmin, m[2i+1]) (the 6-bit unpack of the 12 scale
        // bytes s: with j = k mod 4, k < 4 takes s[j] & 63 and s[j+4] & 63;
        // k >= 4 takes the low / high nibble of s[j+8] with the top bits of
        // s[j] / s[j+4]); the others arrive by shuffle.
        const uint32_t hd = *reinterpret_cast<const uint32_t*>(b);
        const uint32_t k = 2u * i + (t >> 1), j = k & 3u;
        const uint32_t b0 = b[4u + j], b1 = b[8u + j], b2 = b[12u + j];
        const bool mn = (t & 1u) != 0u;
        const uint32_t lo = mn ? b1 : b0;
        const uint32_t sv = k < 4u ? (lo & 63u) : ((mn ? (b2 >> 4) : (b2 & 15u)) | ((lo >> 6) << 4));
        const float sc = __fmul_rn(h2f(mn ? (hd >> 16) : (hd & 0xffffu)), small_uint(sv));
        const float f = mn ? -sc : sc;
        const uint32_t g = lane & ~3u;
        const float da0 = __shfl_sync(0xffffffffu, f, g), ndm0 = __shfl_sync(0xffffffffu, f, g | 1u);
        const float da1 = __shfl_sync(0xffffffffu, f, g | 2u), ndm1 = __shfl_sync(0xffffffffu, f, g | 3u);
        const float bias = 8388608.0f;  // 2^23
        gl_fma_acc<WBF16>(da0, w0 & 0x0F0F0F0Fu, bias, ndm0, x, acc);
        gl_fma_acc<WBF16>(da0, w1 & 0x0F0F0F0Fu, bias, ndm0, x + 4, acc);
        gl_fma_acc<WBF16>(da1, (w0 >> 4) & 0x0F0F0F0Fu, bias, ndm1, x + 8, acc);
        gl_fma_acc<WBF16>(da1, (w1 >> 4) & 0x0F0F0F0Fu, bias, ndm1, x + 12, acc);
    }
    struct U {
        uint32_t w0, w1;
        float da0, ndm0, da1, ndm1;
    };
    __device__ __forceinline__ static U prep(const uint8_t* in, uint32_t u, uint32_t lane) {
        const uint32_t s = u & 15u, i = s >> 2, t = s & 3u;
        const uint8_t* b = in + (u >> 4) * 144u;
        U v;
        v.w0 = *reinterpret_cast<const uint32_t*>(b + 16u + 32u * i + 4u * t);
        v.w1 = *reinterpret_cast<const uint32_t*>(b + 32u + 32u * i + 4u * t);
        const uint32_t hd = *reinterpret_cast<const uint32_t*>(b);
        const uint32_t k = 2u * i + (t >> 1), j = k & 3u;
        const uint32_t b0 = b[4u + j], b1 = b[8u + j], b2 = b[12u + j];
        const bool mn = (t & 1u) != 0u;
        const uint32_t lo = mn ? b1 : b0;
        const uint32_t sv = k < 4u ? (lo & 63u) : ((mn ? (b2 >> 4) : (b2 & 15u)) | ((lo >> 6) << 4));
        const float sc = __fmul_rn(h2f(mn ? (hd >> 16) : (hd & 0xffffu)), small_uint(sv));
        const float f = mn ? -sc : sc;
        const uint32_t g = lane & ~3u;
        v.da0 = __shfl_sync(0xffffffffu, f, g);
        v.ndm0 = __shfl_sync(0xffffffffu, f, g | 1u);
        v.da1 = __shfl_sync(0xffffffffu, f, g | 2u);
        v.ndm1 = __shfl_sync(0xffffffffu, f, g | 3u);
        return v;
    }
    template <bool WBF16>
    __device__ __forceinline__ static void run(const U& s, int r, float2& w01, float2& w23) {
        const uint32_t c = ((r & 1) ? s.w1 : s.w0) >> ((r & 2) ? 4 : 0) & 0x0F0F0F0Fu;
        const float a = r < 2 ? s.da0 : s.da1, m = r < 2 ? s.ndm0 : s.ndm1;
        const float2 aa = make_float2(a, a), cc = make_float2(m, m);
        w01 = gl_round<WBF16>(gm_fma2(aa, gm_bytes_minus2<0>(c, 8388608.0f), cc));
        w23 = gl_round<WBF16>(gm_fma2(aa, gm_bytes_minus2<2>(c, 8388608.0f), cc));
    }
};

// gguf:q6_k: unit u = 16 b + s of block b: half h = s >> 3 and l0 = 4 (s & 7);
// run r holds elements 128h + l0 + 32r .. +3, whose low nibbles are low
// bytes 64h + l0 (runs 0, 2: low / high nibble) and 64h + 32 + l0 (runs 1,
// 3), whose 2-bit high parts are bits 2r of high bytes 32h + l0, and whose
// scale is scales[8h + 2r + (l0 >= 16)].
template <>
struct Gl<KF_Q6_K> {
    static constexpr bool kLean = true;
    __device__ __forceinline__ static uint32_t col(uint32_t u, int r) {
        const uint32_t s = u & 15u;
        return 256u * (u >> 4) + 128u * (s >> 3) + 4u * (s & 7u) + 32u * r;
    }
    template <bool WBF16>
    __device__ __forceinline__ static void unit(const uint8_t* in, uint32_t u, uint32_t lane, const float* x,
                                                float2& acc) {
        const uint32_t s = u & 15u, h = s >> 3, l0 = 4u * (s & 7u);
        const uint32_t off = (u >> 4) * 210u;  // even: every field below is at an even offset
        const uint32_t a = lds_4h(in, off + 64u * h + l0), c = lds_4h(in, off + 64u * h + 32u + l0);
        const uint32_t q = lds_4h(in, off + 128u + 32u * h + l0);
        // lane s & 3 of the group forms the scale of run s & 3
        const float d = h2f(*reinterpret_cast<const uint16_t*>(in + off + 208u));
        const float dl = __fmul_rn(d, i8_float(in[off + 192u + 8u * h + ((s >> 2) & 1u) + 2u * (s & 3u)]));
        const uint32_t g = lane & ~3u;
        const float ds0 = __shfl_sync(0xffffffffu, dl, g), ds1 = __shfl_sync(0xffffffffu, dl, g | 1u);
        const float ds2 = __shfl_sync(0xffffffffu, dl, g | 2u), ds3 = __shfl_sync(0xffffffffu, dl, g | 3u);
        const float bias = 8388640.0f;  // 2^23 + 32
        gl_mul_acc<WBF16>(ds0, (a & 0x0F0F0F0Fu) | ((q & 0x03030303u) << 4), bias, x, acc);
        gl_mul_acc<WBF16>(ds1, (c & 0x0F0F0F0Fu) | ((q & 0x0C0C0C0Cu) << 2), bias, x + 4, acc);
        gl_mul_acc<WBF16>(ds2, ((a >> 4) & 0x0F0F0F0Fu) | (q & 0x30303030u), bias, x + 8, acc);
        gl_mul_acc<WBF16>(ds3, ((c >> 4) & 0x0F0F0F0Fu) | ((q >> 2) & 0x30303030u), bias, x + 12, acc);
    }
    struct U {
        uint32_t a, c, q;
        float ds0, ds1, ds2, ds3;
    };
    __device__ __forceinline__ static U prep(const uint8_t* in, uint32_t u, uint32_t lane) {
        const uint32_t s = u & 15u, h = s >> 3, l0 = 4u * (s & 7u);
        const uint32_t off = (u >> 4) * 210u;
        U v;
        v.a = lds_4h(in, off + 64u * h + l0);
        v.c = lds_4h(in, off + 64u * h + 32u + l0);
        v.q = lds_4h(in, off + 128u + 32u * h + l0);
        const float d = h2f(*reinterpret_cast<const uint16_t*>(in + off + 208u));
        const float dl = __fmul_rn(d, i8_float(in[off + 192u + 8u * h + ((s >> 2) & 1u) + 2u * (s & 3u)]));
        const uint32_t g = lane & ~3u;
        v.ds0 = __shfl_sync(0xffffffffu, dl, g);
        v.ds1 = __shfl_sync(0xffffffffu, dl, g | 1u);
        v.ds2 = __shfl_sync(0xffffffffu, dl, g | 2u);
        v.ds3 = __shfl_sync(0xffffffffu, dl, g | 3u);
        return v;
    }
    template <bool WBF16>
    __device__ __forceinline__ static void run(const U& s, int r, float2& w01, float2& w23) {
        uint32_t code;
        float d;
        if (r == 0) {
            code = (s.a & 0x0F0F0F0Fu) | ((s.q & 0x03030303u) << 4);
            d = s.ds0;
        } else if (r == 1) {
            code = (s.c & 0x0F0F0F0Fu) | ((s.q & 0x0C0C0C0Cu) << 2);
            d = s.ds1;
        } else if (r == 2) {
            code = ((s.a >> 4) & 0x0F0F0F0Fu) | (s.q & 0x30303030u);
            d = s.ds2;
        } else {
            code = ((s.c >> 4) & 0x0F0F0F0Fu) | ((s.q >> 2) & 0x30303030u);
            d = s.ds3;
        }
        const float2 dd = make_float2(d, d);
        const float bias = 8388640.0f;  // 2^23 + 32
        w01 = gl_round<WBF16>(gm_mul2(dd, gm_bytes_minus2<0>(code, bias)));
        w23 = gl_round<WBF16>(gm_mul2(dd, gm_bytes_minus2<2>(code, bias)));
    }
};

// XR: warp iterations (units) per lane per row, 1, 2 or 4 (K <= 4096 XR);
// at most RBM rows per stage (p.rows_per_stage).
template <int F, int XR, bool WBF16>
__global__ void __launch_bounds__(kBlockThreads, 2) k_gemvl(const MvParams p) {
    using G = Gl<F>;
    constexpr uint32_t RBM = XR >= 4 ? 2u : kGlMaxRows;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t slot = static_cast<uint32_t>(p.slot), rb = static_cast<uint32_t>(p.rows_per_stage);
    SmemHdr& H = *reinterpret_cast<SmemHdr*>(smem + kGlStages * slot);
    GlShared& R = *reinterpret_cast<GlShared*>(smem + kGlStages * slot + kHdrBytes);
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t nit = static_cast<uint32_t>(p.K / kGlIter);
    const uint32_t cw = (nit + XR - 1) / XR;  // warps with iterations (at most 8)
    const uint32_t rowb = static_cast<uint32_t>(p.bpr * p.w.S);  // a multiple of 16
    const uint64_t nblk = p.gt[p.nt - 1].blk_end;
    // row block -> (tensor, first row, rows): tensor t holds blocks
    // [gt[t-1].blk_end, gt[t].blk_end)
    auto locate = [&](uint64_t blk, int& t, uint64_t& r0, uint32_t& nr) {
        t = 0;
        while (t + 1 < p.nt && blk >= p.gt[t].blk_end) ++t;
        r0 = (blk - (t > 0 ? p.gt[t - 1].blk_end : 0u)) * rb;
        const uint64_t left = p.gt[t].rows - r0;
        nr = static_cast<uint32_t>(left < rb ? left : rb);
    };
    if (tid == 0) {
        for (int s = 0; s < kGlStages; ++s) {
            mbar_init(&H.full[s], 1);
            mbar_init(&H.empty[s], cw);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < kGlStages) R.cnt[tid] = 0u;
    // warm L2 with this CTA's first row block (the weights are launch
    // parameters; the activations, which the previous kernel may write, are
    // read after the wait)
    if (tid == kThreads && blockIdx.x < nblk) {
        int t;
        uint64_t r0;
        uint32_t nr;
        locate(blockIdx.x, t, r0, nr);
        const uint32_t bytes = nr * rowb;
        prefetch_l2(p.gt[t].x + r0 * rowb, bytes < 32768u ? bytes : 32768u);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    if (tid >= kThreads) {  // producer: one bulk copy per row block
        if (tid != kThreads) return;
        int issued = 0;
        bool fault = false;
        for (uint64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x, ++issued) {
            const int s = issued % kGlStages;
            if (issued >= kGlStages &&
                !mbar_wait_bounded(&H.empty[s], static_cast<uint32_t>(((issued / kGlStages) - 1) & 1))) {
                fault = true;
                break;
            }
            int t;
            uint64_t r0;
            uint32_t nr;
            locate(blk, t, r0, nr);
            const uint32_t bytes = nr * rowb;
            mbar_arrive_expect_tx(&H.full[s], bytes);
            bulk_load(smem + static_cast<uint32_t>(s) * slot, p.gt[t].x + r0 * rowb, bytes, &H.full[s]);
        }
        if (fault) {
            atomicOr(p.fault, 1u);
            for (int j = issued - kGlStages; j < issued; ++j)
                if (j >= 0) mbar_wait_bounded(&H.full[j % kGlStages], static_cast<uint32_t>((j / kGlStages) & 1));
        }
        return;
    }
    if (warp >= cw) return;

    // this lane's activations: run r of unit 32 (XR warp + j) + lane
    float xv[XR][16];
#pragma unroll
    for (int j = 0; j < XR; ++j) {
        const uint32_t it = warp * XR + j;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            uint32_t lo = 0u, hi = 0u;
            if (it < nit) {
                const uint16_t* xp = p.x + G::col(32u * it + lane, r);
                if (p.xvec) {
                    const uint2 t2 = __ldg(reinterpret_cast<const uint2*>(xp));
                    lo = t2.x;
                    hi = t2.y;
                } else {
                    lo = static_cast<uint32_t>(__ldg(xp)) | (static_cast<uint32_t>(__ldg(xp + 1)) << 16);
                    hi = static_cast<uint32_t>(__ldg(xp + 2)) | (static_cast<uint32_t>(__ldg(xp + 3)) << 16);
                }
            }
            xv[j][4 * r] = bf16_lo(lo);
            xv[j][4 * r + 1] = bf16_hi(lo);
            xv[j][4 * r + 2] = bf16_lo(hi);
            xv[j][4 * r + 3] = bf16_hi(hi);
        }
    }

    int n = 0;
    for (uint64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x, ++n) {
        const int s = n % kGlStages;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&H.full[s], static_cast<uint32_t>((n / kGlStages) & 1)))) {
            if (lane == 0) atomicOr(p.fault, 2u);
            return;
        }
        int t;
        uint64_t r0;
        uint32_t nr;
        locate(blk, t, r0, nr);
        const uint8_t* in = smem + static_cast<uint32_t>(s) * slot;
        float2 acc[RBM];
#pragma unroll
        for (uint32_t r = 0; r < RBM; ++r) acc[r] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < XR; ++j) {
            const uint32_t it = warp * XR + j;
            if (it < nit) {
#pragma unroll
                for (uint32_t r = 0; r < RBM; ++r)
                    if (r < nr) G::template unit<WBF16>(in + r * rowb, 32u * it + lane, lane, xv[j], acc[r]);
            }
        }
        // the RBM row sums over the warp: halve the rows a lane keeps at lane
        // offsets 16, 8, 4 (RBM = 8) or 16 (RBM = 2), then add over the rest;
        // lane 4k (RBM = 8) or lane 16k (RBM = 2) ends with row k
        float v[RBM];
#pragma unroll
        for (uint32_t r = 0; r < RBM; ++r) v[r] = __fadd_rn(acc[r].x, acc[r].y);
        uint32_t keep = RBM, o = 16u;
#pragma unroll
        for (; keep > 1u; keep >>= 1, o >>= 1) {
            const bool up = (lane & o) != 0u;
#pragma unroll
            for (uint32_t i = 0; i < keep / 2u; ++i) {
                const float mine = up ? v[keep / 2u + i] : v[i], other = up ? v[i] : v[keep / 2u + i];
                v[i] = __fadd_rn(mine, __shfl_xor_sync(0xffffffffu, other, o));
            }
        }
#pragma unroll
        for (; o > 0u; o >>= 1) v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], o));
        constexpr uint32_t kStep = 32u / RBM;  // lanes per row after the halving
        const uint32_t myrow = (RBM == 8u) ? (lane >> 2) : (lane >> 4);
        if (lane % kStep == 0u && myrow < nr) R.red[s][myrow][warp] = v[0];
        __syncwarp();
        bool last = false;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&R.cnt[s], 1u) == cw - 1u;
        }
        last = __shfl_sync(0xffffffffu, last ? 1u : 0u, 0) != 0u;
        if (last) {  // the stage's last warp adds each row's partials in warp order
            __threadfence_block();
            if (lane < nr) {
                float y = R.red[s][lane][0];
                for (uint32_t w = 1; w < cw; ++w) y = __fadd_rn(y, R.red[s][lane][w]);
                if (p.out_bf16)
                    static_cast<__nv_bfloat16*>(p.gt[t].y)[r0 + lane] = __float2bfloat16_rn(y);
                else
                    static_cast<float*>(p.gt[t].y)[r0 + lane] = y;
            }
            __syncwarp();
            if (lane == 0) R.cnt[s] = 0u;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&H.empty[s]);
    }
}

// ---------------------------------------------------------------------------
// Activations in shared memory, lean decoders: k_gemvm.  For the formats of
// k_gemvl, 1 to 8 activation rows, K a multiple of 512 up to 16384 with X
// and three slots of 4 rows fitting shared memory, 16-byte-aligned rows (the
// host takes it for 2 to 8 rows, and for one row when K > 4096).  One CTA
// per SM (16 warps; 8 for 5 to 8 activation rows, whose accumulators take
// more registers); a ring of 3 slots, each holding rb whole weight rows
// staged by one bulk copy, which the last warp to finish a slot issues for
// the slot's next row block (no producer warp).  The warps first convert X
// to binary32 in shared memory, in lane-unit order (iteration it,
// activation row m, run r, lane: 4 floats), so that a warp reads the 4
// activations of one run of its 32 units with one 16-byte load per lane,
// without bank conflicts.  Warp (it, g) takes the units of iteration it
// (32 it + lane) of every row, for all the activation rows, and the row
// quads g, g + rg, ... of each stage (with more iterations than warps,
// every nwi-th iteration of the row from it): it decodes one unit of 4
// weight rows at a time (the unit's fields first, then run by run the 4 x 4
// weights)
// and adds them times the MP activation runs into 4 MP independent FMA-pair
// chains.  Per weight that is one decode, M multiply-adds (the FMA pipe)
// and, 4 rows sharing each activation load, M bytes of X read from shared
// memory.  A warp reduces its 4 MP sums together (reduce-scatter, then a
// butterfly) and stores one partial per (row, activation row, warp along
// the row); the last warp of the stage adds each output's partials in
// order.  Products and sums are binary32; W is the exact decode (or its
// bfloat16 rounding), formed exactly as the decode kernels do.
// ---------------------------------------------------------------------------
// Warps of a CTA for a kernel of mp activation rows.
__host__ __device__ constexpr uint32_t gm_warps(uint32_t mp) { return mp > 4u ? 8u : 16u; }
constexpr int kGmStages = 3;
constexpr uint32_t kGmQuad = 4;                  // weight rows per warp pass
constexpr uint32_t kGmSmemMax = 227u * 1024u;    // dynamic shared memory of one CTA per SM
constexpr uint32_t kGmHdrBytes = 128;

struct GmHdr {
    uint64_t full[kGmStages];
    uint32_t cnt[kGmStages];  // warps that stored their partials of the stage
};
static_assert(sizeof(GmHdr) <= kGmHdrBytes, "GmHdr layout");

// Warps along a row: one per iteration, or, when there are more iterations
// than warps, the largest divisor nwi of nit that is at most the warp count
// (each such warp takes iterations i0, i0 + nwi, ...: nit / nwi of them).
__host__ __device__ constexpr uint32_t gm_row_warps(uint32_t nit, uint32_t mp) {
    uint32_t d = nit < gm_warps(mp) ? nit : gm_warps(mp);
    while (d > 1u && nit % d != 0u) --d;
    return d;
}
// Row groups of a launch: each row quad takes gm_row_warps warps.
__host__ __device__ constexpr uint32_t gm_row_groups(uint32_t nit, uint32_t mp) {
    return gm_warps(mp) / gm_row_warps(nit, mp);
}

// Dynamic shared memory: the stage slots, X as binary32, the header, and
// the partial sums (stage, row, activation row, warp along the row).
__host__ __device__ constexpr size_t gm_smem_bytes(uint32_t slot, uint32_t mp, uint64_t K, uint32_t rb) {
    return static_cast<size_t>(kGmStages) * slot + static_cast<size_t>(mp) * K * 4u + kGmHdrBytes +
           static_cast<size_t>(kGmStages) * rb * mp * gm_row_warps(static_cast<uint32_t>(K / kGlIter), mp) * 4u;
}

// MI: a warp may take several iterations (K / 512 above the warp count);
// without it every warp takes exactly one.
template <int F, int MP, bool MI, bool WBF16>
__global__ void __launch_bounds__(gm_warps(MP) * 32, 1) k_gemvm(const MvParams p) {
    using G = Gl<F>;
    constexpr uint32_t NT = gm_warps(MP) * 32u, NV = kGmQuad * MP;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t slot = static_cast<uint32_t>(p.slot), rb = static_cast<uint32_t>(p.rows_per_stage);
    const uint32_t nit = static_cast<uint32_t>(p.K / kGlIter);
    const uint32_t nwi = gm_row_warps(nit, MP), rg = gm_row_groups(nit, MP), wu = rg * nwi;
    const uint32_t xbytes = static_cast<uint32_t>(MP * p.K * 4u);
    float4* xs = reinterpret_cast<float4*>(smem + kGmStages * slot);
    GmHdr& H = *reinterpret_cast<GmHdr*>(smem + kGmStages * slot + xbytes);
    float* red = reinterpret_cast<float*>(smem + kGmStages * slot + xbytes + kGmHdrBytes);
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t rowb = static_cast<uint32_t>(p.bpr * p.w.S);  // a multiple of 16
    const uint64_t N = p.n_rows, nblk = (N + rb - 1u) / rb;
    // row block b (first row b rb) into stage s
    auto stage_in = [&](uint64_t b, int s) {
        const uint64_t r0 = b * rb;
        const uint32_t bytes = static_cast<uint32_t>(N - r0 < rb ? N - r0 : rb) * rowb;
        mbar_arrive_expect_tx(&H.full[s], bytes);
        bulk_load(smem + static_cast<uint32_t>(s) * slot, p.w.x + r0 * rowb, bytes, &H.full[s]);
    };
    if (tid == 0) {
        for (int s = 0; s < kGmStages; ++s) {
            mbar_init(&H.full[s], 1);
            H.cnt[s] = 0u;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // warm L2 with this CTA's first row block (the weights are launch
        // parameters; the activations, which the previous kernel may write,
        // are read after the wait)
        if (blockIdx.x < nblk) {
            const uint64_t r0 = static_cast<uint64_t>(blockIdx.x) * rb;
            const uint32_t bytes = static_cast<uint32_t>(N - r0 < rb ? N - r0 : rb) * rowb;
            prefetch_l2(p.w.x + r0 * rowb, bytes < 32768u ? bytes : 32768u);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();
    if (tid == 0)
        for (int s = 0; s < kGmStages; ++s)
            if (blockIdx.x + static_cast<uint64_t>(s) * gridDim.x < nblk)
                stage_in(blockIdx.x + static_cast<uint64_t>(s) * gridDim.x, s);

    // X as binary32 in lane-unit order: entry e = ((it MP + m) 4 + r) 32 + l
    // holds activations col(32 it + l, r) .. +3 of row m (zeros for m >= M);
    // kGmXIn entries per thread are loaded before any is stored, so that
    // their global reads overlap
    const uint32_t nx = MP * nit * 128u;
    constexpr uint32_t kGmXIn = 8;
    for (uint32_t e0 = tid; e0 < nx; e0 += NT * kGmXIn) {
        uint2 xv[kGmXIn];
#pragma unroll
        for (uint32_t j = 0; j < kGmXIn; ++j) {
            const uint32_t e = e0 + j * NT;
            const uint32_t l = e & 31u, r = (e >> 5) & 3u, q = e >> 7, it = q / MP, m = q % MP;
            xv[j] = make_uint2(0u, 0u);
            if (e < nx && m < static_cast<uint32_t>(p.m)) {
                const uint16_t* xp =
                    p.x + static_cast<uint64_t>(m) * p.K + G::col(32u * it + l, static_cast<int>(r));
                if (p.xvec) {
                    xv[j] = __ldg(reinterpret_cast<const uint2*>(xp));
                } else {
                    xv[j].x = static_cast<uint32_t>(__ldg(xp)) | (static_cast<uint32_t>(__ldg(xp + 1)) << 16);
                    xv[j].y = static_cast<uint32_t>(__ldg(xp + 2)) | (static_cast<uint32_t>(__ldg(xp + 3)) << 16);
                }
            }
        }
#pragma unroll
        for (uint32_t j = 0; j < kGmXIn; ++j) {
            const uint32_t e = e0 + j * NT;
            if (e < nx) xs[e] = make_float4(bf16_lo(xv[j].x), bf16_hi(xv[j].x), bf16_lo(xv[j].y), bf16_hi(xv[j].y));
        }
    }
    __syncthreads();
    if (warp >= wu) return;

    const uint32_t i0 = warp % nwi, g = warp / nwi;
    int n = 0;
    for (uint64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x, ++n) {
        const int s = n % kGmStages;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&H.full[s], static_cast<uint32_t>((n / kGmStages) & 1)))) {
            // give copies already issued to the next slots time to land
            // before the CTA's shared memory is released
            if (lane == 0) {
                atomicOr(p.fault, 2u);
                for (int j = n + 1; j < n + kGmStages; ++j)
                    if (blockIdx.x + static_cast<uint64_t>(j) * gridDim.x < nblk)
                        mbar_wait_bounded(&H.full[j % kGmStages], static_cast<uint32_t>((j / kGmStages) & 1));
            }
            __syncwarp();
            return;
        }
        const uint64_t r0 = blk * rb;
        const uint32_t nr = static_cast<uint32_t>(N - r0 < rb ? N - r0 : rb);
        const uint8_t* in = smem + static_cast<uint32_t>(s) * slot;
        // row quads of this warp (rows past nr decode stale slot bytes;
        // their sums are never read)
        for (uint32_t qb = kGmQuad * g; qb < rb; qb += kGmQuad * rg) {
            float2 acc[kGmQuad][MP];
#pragma unroll
            for (uint32_t k = 0; k < kGmQuad; ++k)
#pragma unroll
                for (uint32_t mm = 0; mm < MP; ++mm) acc[k][mm] = make_float2(0.0f, 0.0f);
            // the quad's units of iteration it, times the activation runs
            auto one_it = [&](uint32_t it) {
                const float4* xw = xs + it * MP * 128u + lane;  // activation row m, run r: + 128 m + 32 r
                const uint32_t u = 32u * it + lane;
                typename G::U su[kGmQuad];
#pragma unroll
                for (uint32_t k = 0; k < kGmQuad; ++k) su[k] = G::prep(in + (qb + k) * rowb, u, lane);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    float2 wv[kGmQuad][2];
#pragma unroll
                    for (uint32_t k = 0; k < kGmQuad; ++k) G::template run<WBF16>(su[k], r, wv[k][0], wv[k][1]);
#pragma unroll
                    for (uint32_t mm = 0; mm < MP; ++mm) {
                        const float4 xv = xw[128u * mm + 32u * static_cast<uint32_t>(r)];
                        const float2 x01 = make_float2(xv.x, xv.y), x23 = make_float2(xv.z, xv.w);
#pragma unroll
                        for (uint32_t k = 0; k < kGmQuad; ++k) {
                            acc[k][mm] = gm_fma2(x01, wv[k][0], acc[k][mm]);
                            acc[k][mm] = gm_fma2(x23, wv[k][1], acc[k][mm]);
                        }
                    }
                }
            };
            if constexpr (MI) {
#pragma unroll 1
                for (uint32_t it = i0; it < nit; it += nwi) one_it(it);
            } else {
                one_it(i0);
            }
            // the NV sums over the warp: halve the values a lane keeps at
            // lane offsets 16, 8, ... then add over the rest; lane
            // (32 / NV) i ends with value i = k MP + mm
            float v[NV];
#pragma unroll
            for (uint32_t k = 0; k < kGmQuad; ++k)
#pragma unroll
                for (uint32_t mm = 0; mm < MP; ++mm) v[k * MP + mm] = __fadd_rn(acc[k][mm].x, acc[k][mm].y);
            uint32_t keep = NV, o = 16u;
#pragma unroll
            for (; keep > 1u; keep >>= 1, o >>= 1) {
                const bool up = (lane & o) != 0u;
#pragma unroll
                for (uint32_t i = 0; i < keep / 2u; ++i) {
                    const float mine = up ? v[keep / 2u + i] : v[i], other = up ? v[i] : v[keep / 2u + i];
                    v[i] = __fadd_rn(mine, __shfl_xor_sync(0xffffffffu, other, o));
                }
            }
#pragma unroll
            for (; o > 0u; o >>= 1) v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], o));
            constexpr uint32_t kStep = 32u / NV;
            if (lane % kStep == 0u) {
                const uint32_t vi = lane / kStep, k = vi / MP, mm = vi % MP;
                red[((static_cast<uint32_t>(s) * rb + qb + k) * MP + mm) * nwi + i0] = v[0];
            }
        }
        __syncwarp();
        bool last = false;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&H.cnt[s], 1u) == wu - 1u;
        }
        last = __shfl_sync(0xffffffffu, last ? 1u : 0u, 0) != 0u;
        if (last) {
            // the stage's last warp: every warp is done with the slot and its
            // partials; add each output's partials in iteration order, then
            // stage the slot's next row block
            __threadfence_block();
            const uint32_t no = nr * static_cast<uint32_t>(p.m);
            for (uint32_t o2 = lane; o2 < no; o2 += 32u) {
                const uint32_t row = o2 % nr, m = o2 / nr;
                const float* pr = red + ((static_cast<uint32_t>(s) * rb + row) * MP + m) * nwi;
                float y = pr[0];
                for (uint32_t w = 1; w < nwi; ++w) y = __fadd_rn(y, pr[w]);
                const uint64_t yi = static_cast<uint64_t>(m) * N + r0 + row;
                if (p.out_bf16)
                    static_cast<__nv_bfloat16*>(p.y)[yi] = __float2bfloat16_rn(y);
                else
                    static_cast<float*>(p.y)[yi] = y;
            }
            __syncwarp();
            if (lane == 0) {
                H.cnt[s] = 0u;
                const uint64_t nb = blk + static_cast<uint64_t>(kGmStages) * gridDim.x;
                if (nb < nblk) {
                    fence_proxy_async_smem();  // the slot's reads before the copy that overwrites it
                    stage_in(nb, s);
                }
            }
            __syncwarp();
        }
    }
}

}  // namespace

// Fused kernel of decode family F for a launch variant (used by the
// per-format instantiation files; see MvVariant in ndq_internal.h).
template <int F>
MvKernelFn matvec_kernel(int variant) {
    if (variant >= kMvMulti) {
        if constexpr (Gl<F>::kLean) {
            switch (variant - kMvMulti) {
                case 0: return k_gemvm<F, 1, false, false>;
                case 1: return k_gemvm<F, 1, false, true>;
                case 2: return k_gemvm<F, 1, true, false>;
                case 3: return k_gemvm<F, 1, true, true>;
                case 4: return k_gemvm<F, 2, false, false>;
                case 5: return k_gemvm<F, 2, false, true>;
                case 6: return k_gemvm<F, 2, true, false>;
                case 7: return k_gemvm<F, 2, true, true>;
                case 8: return k_gemvm<F, 4, false, false>;
                case 9: return k_gemvm<F, 4, false, true>;
                case 10: return k_gemvm<F, 4, true, false>;
                case 11: return k_gemvm<F, 4, true, true>;
                case 12: return k_gemvm<F, 8, false, false>;
                case 13: return k_gemvm<F, 8, false, true>;
                case 14: return k_gemvm<F, 8, true, false>;
                default: return k_gemvm<F, 8, true, true>;
            }
        }
        return nullptr;
    }
    if (variant >= kMvLean) {
        if constexpr (Gl<F>::kLean) {
            switch (variant - kMvLean) {
                case 0: return k_gemvl<F, 1, false>;
                case 1: return k_gemvl<F, 1, true>;
                case 2: return k_gemvl<F, 2, false>;
                case 3: return k_gemvl<F, 2, true>;
                case 4: return k_gemvl<F, 4, false>;
                default: return k_gemvl<F, 4, true>;
            }
        }
        return nullptr;
    }
    switch (variant) {
        case kMvOneRowF32: return k_gemv1<F, true>;
        case kMvOneRowF32Any: return k_gemv1<F, false>;
        case kMvRowsBf16: return k_matvec<F, kMvMaxRows, true, kMvXBf16>;
        case kMvRowsGlobal: return k_matvec<F, kMvMaxRows, true, kMvXGlobal>;
        default: return k_matvec<F, kMvMaxRows, false, kMvXGlobal>;
    }
}

}  // namespace ndq
