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

// Accumulate this thread's chunks of one staged unit into acc[m]: the
// thread's row group g = tid / (256/R) owns row g of the unit, whose nb
// blocks hold nb*CPB chunks; the group's threads take them in turn.
template <int F, bool PH, int MT>
__device__ __forceinline__ void mv_tile(const MvStage& st, const uint8_t* in, const Ctx& x, uint32_t tid,
                                        const MvParams& p, float* acc) {
    using Fm = Fmt<F>;
    constexpr int CE = Fm::CE;
    const uint32_t gsize = kThreads / static_cast<uint32_t>(p.rows_per_stage);
    const uint32_t g = tid / gsize;
    if (g >= st.nrows) return;
    const uint32_t per_row = st.nb * static_cast<uint32_t>(Fm::CPB);
    const uint32_t ph = PH ? st.phase : 0u;
    const uint16_t* xg = p.x + st.k0;
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
        const uint64_t col = static_cast<uint64_t>(CE) * j;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (MT == 1 || m < p.m) {
                const uint16_t* xr = xg + static_cast<uint64_t>(m) * p.K + col;
                uint32_t xb[CE / 2];
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
                // two interleaved chains (even / odd elements) for latency
                float a0 = acc[m], a1 = 0.0f;
#pragma unroll
                for (int i = 0; i < CE / 2; ++i) {
                    a0 = __fmaf_rn(bf16_lo(xb[i]), v[2 * i], a0);
                    a1 = __fmaf_rn(bf16_hi(xb[i]), v[2 * i + 1], a1);
                }
                acc[m] = __fadd_rn(a0, a1);
            }
        }
    }
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
            const uint64_t left = p.bpr - sb;
            const uint32_t nb = static_cast<uint32_t>(left < seg ? left : seg);
            const uint64_t b0 = row0 * p.bpr + sb;
            const uint8_t* src = t.x + b0 * t.S;
            const uint32_t phase = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
            const uint32_t bytes = (phase + nrows * nb * t.S + 15u) & ~15u;
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
// loads.
template <int F, int MT, bool ALIGNED>
__global__ void __launch_bounds__(kBlockThreads, 2) k_matvec(const MvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* inbuf = smem;
    SmemHdr& H = *reinterpret_cast<SmemHdr*>(smem + kStages * kInStride);
    MvShared& S = *reinterpret_cast<MvShared*>(smem + kStages * kInStride + kHdrBytes);
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
    __syncthreads();

    if (tid >= kThreads) {  // producer warp
        if (tid == kThreads) mv_producer(p, H, S, inbuf);
        return;
    }

    const uint32_t lane = tid & 31u, warp = tid >> 5;
    const DevTensor& t = p.w;
    const Ctx base{&H, nullptr, t.divs, 0, t.blocks_per_div, p.grids, code_count(t), 0, 0};
    const uint64_t R = static_cast<uint64_t>(p.rows_per_stage);
    const uint64_t seg = R > 1 ? p.bpr : static_cast<uint64_t>(t.bpt);
    const uint64_t units = (p.n_rows + R - 1) / R;
    const uint32_t gwarps = static_cast<uint32_t>(kConsumerWarps / R);  // warps per row group
    const uint32_t g = warp / gwarps;                                    // this warp's row group
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
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
            mv_tile<F, !ALIGNED, MT>(st, in, x, tid, p, acc);
            if (st.last && g < st.nrows) {
                // warp partials, then the last warp of the row group adds the
                // group's partials in warp order
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (MT == 1 || m < p.m) {
                        float v = acc[m];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                        if (lane == 0) S.red[s][warp][m] = v;
                    }
                    acc[m] = 0.0f;
                }
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

}  // namespace

// Fused kernel of decode family F for a launch variant (used by the
// per-format instantiation files): 0 = aligned, one activation row;
// 1 = aligned, up to kMvMaxRows rows; 2 = any alignment, up to kMvMaxRows.
template <int F>
MvKernelFn matvec_kernel(int variant) {
    switch (variant) {
        case 0: return k_matvec<F, 1, true>;
        case 1: return k_matvec<F, kMvMaxRows, true>;
        default: return k_matvec<F, kMvMaxRows, false>;
    }
}

}  // namespace ndq
