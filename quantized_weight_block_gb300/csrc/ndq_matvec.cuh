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
// The CTA layout is the decode kernel's: one producer warp stages payload
// units into the shared-memory ring with bulk copies; 8 consumer warps
// decode 16-element chunks with the same Fmt<F> decoders and accumulate
// against X.  A unit is R = rows_per_stage whole weight rows (K <= 8192/R),
// or, when K > 4096, a segment of up to 8192 elements of one row.  Each CTA
// owns whole units, so a row's partial sums meet in the CTA: the 256/R
// threads of a row group take its chunks in turn; warp shuffles, then one
// partial per warp in shared memory; the last warp of the group to finish
// adds the group's partials in warp order and writes Y.
#pragma once

#include "ndq_device.cuh"

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

}  // namespace

// Fused kernel of decode family F for a launch variant (used by the
// per-format instantiation files; see MvVariant in ndq_internal.h).
template <int F>
MvKernelFn matvec_kernel(int variant) {
    switch (variant) {
        case kMvOneRowF32: return k_gemv1<F, true>;
        case kMvOneRowF32Any: return k_gemv1<F, false>;
        case kMvRowsBf16: return k_matvec<F, kMvMaxRows, true, kMvXBf16>;
        case kMvRowsGlobal: return k_matvec<F, kMvMaxRows, true, kMvXGlobal>;
        default: return k_matvec<F, kMvMaxRows, false, kMvXGlobal>;
    }
}

}  // namespace ndq
