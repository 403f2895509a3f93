// ndq_mmag.cuh -- decode fused into a matrix product with few activation
// rows (M <= 8) on the tcgen05 tensor cores, with the exact (binary32)
// weights, for the formats whose weight is one scale per group of G weights
// times a small integer code: W[n, k] = RN(s[n, g(k)] * c[n, k]) with c exact
// in bfloat16 (gguf:q6_k: s = M(d, scales[j]), c = l + 16h - 32, G = 16;
// gguf:q8_0 and q8_g32_fp16: s = d, c = q, G = 32).
//
//     Y[m, n] = sum_g s[n, g] * P[n, g, m],   P[n, g, m] = sum_{k in g} c[n, k] X[m, k]
//
// The tensor core forms P: the A operand is the codes as bfloat16 (exact),
// the B operand holds X in a staircase so that each group's sum lands in its
// own accumulator column: in a k-step of 64 weights (NG = 64 / G groups),
// row g * MP + m of B holds X[m, k] for the k of group g and zeros elsewhere,
// so the four MMAs of the k-step (K = 16 each, the first one overwriting)
// leave P[., g, m] in TMEM column g * MP + m of the k-step's region.  The
// products c * X are exact in binary32 and each group's sum restarts at
// zero, so every P carries at most 32 terms' rounding; the epilogue then
// adds s * P in binary32 FMAs in k order.  The error stays within the fused
// product's bound 2 (K + 16) 2^-24 sum |X W| (the scale multiplies one
// group's sum instead of each term, which the NInfer page leaves to the
// consuming kernel's choice of association).
//
// Roles (warps), joined only by mbarriers:
//   * 0-15 decode: four threads per weight row, one 16-weight chunk each per
//     k-step: the codes into the A operand (128-byte-swizzled K-major) and
//     the group scales into a small array beside it;
//   * 16-19 epilogue: warp w reads TMEM lanes 32 (w % 4) ..: per k-step the
//     region's NG * MP columns, then Y[m] += s * P in registers;
//   * 20 stages the packed payload (the k_mma producer);
//   * 21 issues the MMAs of a k-step once A and B are full and its TMEM
//     region is free, committing to the stage's free barrier and to the
//     region's full barrier;
//   * 22 writes each k-step's X slices into the staircase (the zeros are
//     written once).
// Split-K over a thread-block cluster as in k_mma.  Every wait is bounded.
#pragma once

#include "ndq_mma.cuh"

namespace ndq {
namespace {

constexpr int kMgEpiWarp = 16;      // warps 16..19: the epilogue
constexpr int kMgProducerWarp = 20;
constexpr int kMgIssueWarp = 21;
constexpr int kMgBWarp = 22;
constexpr int kMgThreads = 23 * 32;
constexpr uint32_t kMgRegions = 8;  // TMEM accumulator regions (k-steps in flight)

// Codes-and-scale decoders: chunk c (16 weights) of a staged span as 8
// bfloat16 pairs of exact codes (natural order), and its group's scale.
template <int F>
struct Gc {
    static constexpr bool kOk = false;
    static constexpr int G = 16;
};

// bfloat16 pairs of bytes (I, I+1) of w (values below 128), minus 160 - off
// = the codes minus `off`: 0x43 | byte is 128 + byte, exact.
template <int I>
__device__ __forceinline__ uint32_t bf16_codes(uint32_t w, uint32_t bias2) {
    const uint32_t t = prmt(w, 0x43434343u, I == 0 ? 0x4140u : 0x4342u);
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(bias2));
    return r;
}

// ---------------------------------------------------------------------------
// Lean codes decoder for gguf:q6_k (one span = one block): the four threads
// of a weight row take the two k-steps 2h, 2h+1 of half h of the block as
// runs of 4 codes that come from aligned 32-bit words: thread t takes l0 =
// 4t and 4t + 16 (low bytes 64h + l0 and 64h + 32 + l0, high bytes 32h +
// l0); runs 0 and 1 (K offsets l0, l0 + 32 of k-step 2h) use the low
// nibbles and high-bit pairs 0, 1, runs 2 and 3 (the same offsets of k-step
// 2h + 1) the high nibbles and pairs 2, 3.  Each run is stored as 8 bytes of
// the A operand (the codes exact in bfloat16); thread t also forms the
// scales 8h + t and 8h + 4 + t, group t of each k-step.  `in` is the row's
// staged span, ph the block's byte phase in it; ok = false (a row past N)
// stores zeros.
// ---------------------------------------------------------------------------
struct TlQ6K {
    static constexpr int KS = 2;  // k-steps per call
    template <bool PH>
    __device__ __forceinline__ static void run(const uint8_t* in, uint32_t ph, uint32_t ks, uint32_t t,
                                               uint8_t* const* aS, float* const* sc, uint32_t r, bool ok) {
        const uint32_t h = ks >> 1;
        const float d = h2f(lds_2<PH>(in, ph + 208u));
        sc[0][4u * r + t] = ok ? __fmul_rn(d, i8_float(in[ph + 192u + 8u * h + t])) : 0.0f;
        sc[1][4u * r + t] = ok ? __fmul_rn(d, i8_float(in[ph + 196u + 8u * h + t])) : 0.0f;
#pragma unroll
        for (uint32_t jj = 0; jj < 2; ++jj) {
            const uint32_t l0 = 4u * t + 16u * jj;
            const uint32_t A = lds_4(in, ph + 64u * h + l0), C = lds_4(in, ph + 64u * h + 32u + l0);
            const uint32_t Q = lds_4(in, ph + 128u + 32u * h + l0);
            const uint32_t c[4] = {(A & 0x0F0F0F0Fu) | ((Q & 0x03030303u) << 4),
                                   (C & 0x0F0F0F0Fu) | ((Q & 0x0C0C0C0Cu) << 2),
                                   ((A >> 4) & 0x0F0F0F0Fu) | (Q & 0x30303030u),
                                   ((C >> 4) & 0x0F0F0F0Fu) | ((Q >> 2) & 0x30303030u)};
#pragma unroll
            for (uint32_t q = 0; q < 4; ++q) {
                const uint32_t k = l0 + 32u * (q & 1u);
                const uint2 v = ok ? make_uint2(bf16_codes<0>(c[q], 0x43204320u), bf16_codes<2>(c[q], 0x43204320u))
                                   : make_uint2(0u, 0u);  // (128 + code) - 160
                *reinterpret_cast<uint2*>(aS[q >> 1] + sw128(r, k >> 3) + 8u * ((k >> 2) & 1u)) = v;
            }
        }
    }
};

template <>
struct Gc<KF_Q6_K> {
    static constexpr bool kOk = true;
    static constexpr int G = 16;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, uint32_t* wb,
                                                 float& sc) {
        const uint32_t off = ph + (c >> 4) * 210u, cc = c & 15u, gi = cc >> 3;
        const float d = h2f(lds_2<PH>(in, off + 208u));
        sc = __fmul_rn(d, i8_float(in[off + 192u + cc]));  // exact: 11 x 8 significant bits
        const uint4 lo = lds_16<false>(in, off + 64u * gi + 16u * (cc & 3u));
        const uint4 hi = lds_16<false>(in, off + 128u + 32u * gi + 16u * (cc & 1u));
        const uint32_t pl = 4u * ((cc >> 2) & 1u), phh = 2u * ((cc >> 1) & 3u);
        const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w}, hw[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t w = ((lw[q] >> pl) & 0x0F0F0F0Fu) | (((hw[q] >> phh) & 0x03030303u) << 4);
            wb[2 * q] = bf16_codes<0>(w, 0x43204320u);  // (128 + code) - 160
            wb[2 * q + 1] = bf16_codes<2>(w, 0x43204320u);
        }
    }
};

template <>
struct Gc<KF_Q8_0> {
    static constexpr bool kOk = true;
    static constexpr int G = 32;
    template <bool PH>
    __device__ __forceinline__ static void chunk(const uint8_t* in, uint32_t ph, uint32_t c, uint32_t* wb,
                                                 float& sc) {
        const uint32_t off = ph + (c >> 1) * 34u;
        sc = h2f(lds_2<PH>(in, off));
        const uint4 q = lds_16<false>(in, off + 2u + 16u * (c & 1u));
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
        const float bias = 8388736.0f;  // 2^23 + 128; XOR 0x80 maps signed to offset-128
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t u = qw[i] ^ 0x80808080u;
            // the exact binary32 codes; their bfloat16 is their top half
            const float2 a = bytes_minus2<0>(u, bias), b = bytes_minus2<2>(u, bias);
            wb[2 * i] = prmt(__float_as_uint(a.x), __float_as_uint(a.y), 0x7632u);
            wb[2 * i + 1] = prmt(__float_as_uint(b.x), __float_as_uint(b.y), 0x7632u);
        }
    }
};

struct MgShared {
    uint64_t efree[kMmaMaxStages];  // the epilogue is done with the stage's scales
    uint64_t dfull[kMgRegions];     // the region's MMAs are complete (tcgen05.commit)
    uint64_t dfree[kMgRegions];     // the epilogue has read the region
};

__host__ __device__ constexpr uint32_t mg_ncol(int ng, uint32_t mp) {
    return static_cast<uint32_t>(ng) * mp < 16u ? 16u : static_cast<uint32_t>(ng) * mp;
}
__host__ __device__ constexpr uint32_t mg_scale_bytes(int ng) { return kMmaRows * 4u * static_cast<uint32_t>(ng); }
// Dynamic shared memory: [A x na][B x nb][scales x na][spans x ns][MmaShared][MgShared].
__host__ __device__ constexpr uint32_t mmag_smem_bytes(uint32_t ncol, int ng, uint32_t span, uint32_t na,
                                                       uint32_t ns, uint32_t nb) {
    return 1024u + na * (kMmaATile + mg_scale_bytes(ng)) + nb * mma_b_tile(ncol) + ns * mma_span_stage(span) + 1024u;
}
__host__ __device__ inline void mmag_stages(uint32_t ncol, int ng, uint32_t span, uint32_t* na, uint32_t* ns,
                                            uint32_t* nb) {
    *na = 2u;
    *ns = 2u;
    for (uint32_t a = 4u; a >= 2u; --a)
        for (uint32_t s = 4u; s >= 2u; --s)
            if (mmag_smem_bytes(ncol, ng, span, a, s, kMmaMaxB) <= kMmaSmemLimit && a * 8u + s > *na * 8u + *ns &&
                (a >= 3u || s <= 3u)) {
                *na = a;
                *ns = s;
            }
    *nb = kMmaMaxB;
}

// TMEM -> registers: N consecutive binary32 columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t* v) {
    if constexpr (N == 2) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(taddr));
    } else if constexpr (N == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                     : "r"(taddr));
    } else if constexpr (N == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                     : "r"(taddr));
    } else {
        static_assert(N % 8 == 0, "tmem_ldn: 2, 4 or a multiple of 8 columns");
#pragma unroll
        for (int i = 0; i < N; i += 8)
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                         : "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]),
                           "=r"(v[i + 5]), "=r"(v[i + 6]), "=r"(v[i + 7])
                         : "r"(taddr + static_cast<uint32_t>(i)));
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// MP: activation rows padded to 1, 2, 4 or 8 (p.bn); p.m_rows <= MP.
template <int F, int MP>
__global__ void __launch_bounds__(kMgThreads, 1) k_mmag(const __grid_constant__ MmaParams p) {
    using Gd = Gc<F>;
    constexpr int G = Gd::G, NG = kMmaK / G, NCU = NG * MP;
    constexpr uint32_t NCOL = mg_ncol(NG, MP);
    constexpr uint32_t kTmemCols = kMgRegions * NCOL < 32u ? 32u : kMgRegions * NCOL;
    extern __shared__ __align__(1024) uint8_t mg_smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mg_smem_raw) + 1023u) & ~uintptr_t(1023));
    const uint32_t na = p.na, nb = p.nb;
    uint8_t* sA = base;
    uint8_t* sB = base + na * kMmaATile;
    float* sS = reinterpret_cast<float*>(sB + nb * mma_b_tile(NCOL));
    uint8_t* sP = reinterpret_cast<uint8_t*>(sS) + na * mg_scale_bytes(NG);
    const uint32_t rstride = p.wbox ? p.wbox : mma_row_stride(p.span_bytes);
    const uint32_t stage_bytes = mma_span_stage(p.span_bytes);
    MmaShared& S = *reinterpret_cast<MmaShared*>(sP + p.ns * stage_bytes);
    MgShared& Q = *reinterpret_cast<MgShared*>(sP + p.ns * stage_bytes + sizeof(MmaShared));
    __shared__ uint32_t s_fault;

    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&S.tmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (uint32_t s = 0; s < p.ns; ++s) {
            mbar_init(&S.full[s], p.wbox ? 1 : 32);
            mbar_init(&S.empty[s], kMmaDecoders / 32);
        }
        for (uint32_t s = 0; s < na; ++s) {
            mbar_init(&S.afull[s], kMmaDecoders / 32);
            mbar_init(&S.sfree[s], 1);
            mbar_init(&Q.efree[s], 4);
        }
        for (uint32_t s = 0; s < nb; ++s) {
            mbar_init(&S.bfull[s], 32);  // one arrival per B-warp lane (cp.async completion)
            mbar_init(&S.bfree[s], 1);
        }
        for (uint32_t r = 0; r < kMgRegions; ++r) {
            mbar_init(&Q.dfull[r], 1);
            mbar_init(&Q.dfree[r], 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid == 32) s_fault = 0u;
    if (tid == kMgProducerWarp * 32 && p.wbox)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.wmap)) : "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    bool fault = false;
    uint64_t sp0, sp1;
    mma_span_range(p, sp0, sp1);
    // (programmatic dependent launch) warm L2 with this CTA's first span of
    // payload rows, then wait for the previous kernel before any read of X
    // or the payload and any write of Y
    if (warp == kMgProducerWarp && sp0 < sp1) {
        const uint64_t kl = p.K - sp0 * p.span_elems;
        const uint32_t span = static_cast<uint32_t>((kl < p.span_elems ? kl : p.span_elems) / Fmt<F>::B * Fmt<F>::S);
        for (uint32_t r = lane; r < kMmaRows; r += 32u) {
            const uint64_t n = static_cast<uint64_t>(blockIdx.x) * kMmaRows + r;
            if (n < p.n_rows) {
                const uint8_t* src = p.w.x + (n * p.bpr + sp0 * p.span_elems / Fmt<F>::B) * Fmt<F>::S;
                const uint32_t ph = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
                prefetch_l2(src - ph, (ph + span + 15u) & ~15u);
            }
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t nk = mma_ksteps(p, sp0, sp1);
    const uint64_t n0 = static_cast<uint64_t>(blockIdx.x) * kMmaRows;
    float y[MP];
#pragma unroll
    for (int m = 0; m < MP; ++m) y[m] = 0.0f;

    if (warp == kMgProducerWarp) {
        mma_producer<F>(p, S, sP, rstride, stage_bytes);
    } else if (warp == kMgBWarp) {
        // zeros everywhere once, then per k-step the X slices of the
        // staircase (row g * MP + m, the 16-byte units of group g) by
        // asynchronous copies that every lane has counted on the stage's
        // full barrier when they land (a unit past X reads no bytes and
        // lands as zeros); nb stages ahead of the MMAs
        for (uint32_t i = lane; i < nb * mma_b_tile(NCOL) / 16u; i += 32u)
            reinterpret_cast<uint4*>(sB)[i] = make_uint4(0u, 0u, 0u, 0u);
        const uint64_t kx = sp0 * p.span_elems;
        for (uint32_t j = 0; j < nk; ++j) {
            const uint32_t b = j % nb;
            if (j >= nb && !__all_sync(0xffffffffu, mbar_wait_bounded(&S.bfree[b], ((j / nb) - 1u) & 1u))) {
                if (lane == 0) {
                    atomicOr(p.fault, 4u);
                    atomicOr(&s_fault, 1u);
                }
                break;
            }
            const uint64_t k0 = kx + static_cast<uint64_t>(kMmaK) * j;
            const uint32_t bS = smem_addr(sB + b * mma_b_tile(NCOL));
            for (uint32_t e = lane; e < static_cast<uint32_t>(MP) * 8u; e += 32u) {
                const uint32_t m = e >> 3, u = e & 7u, g = (8u * u) / static_cast<uint32_t>(G);
                const bool in_x = m < p.m_rows && k0 + 8u * u < p.K;
                const uint16_t* src = in_x ? p.x + m * p.K + k0 + 8u * u : p.x;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(bS + sw128(g * MP + m, u)), "l"(src),
                             "r"(in_x ? 16u : 0u)
                             : "memory");
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(&S.bfull[b])) : "memory");
        }
        asm volatile("cp.async.wait_all;" ::: "memory");  // (no copy of this lane outlives the role)
    } else if (warp == kMgIssueWarp) {
        const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((NCOL >> 3) << 17) | ((kMmaRows >> 4) << 24);
        uint32_t issued = 0;
        for (uint32_t i = 0; i < nk; ++i) {
            const uint32_t a = i % na, ap = (i / na) & 1u, b = i % nb, r = i % kMgRegions;
            bool ok = mbar_wait_bounded(&S.afull[a], ap) && mbar_wait_bounded(&S.bfull[b], (i / nb) & 1u);
            if (ok && i >= kMgRegions) ok = mbar_wait_bounded(&Q.dfree[r], ((i / kMgRegions) - 1u) & 1u);
            if (!__all_sync(0xffffffffu, ok)) {
                fault = true;
                break;
            }
            // (the B stage was written by asynchronous copies of the generic
            // proxy: order them before the tensor core's reads)
            fence_proxy_async_smem();
            tc_fence_after();
            const uint32_t a0 = smem_addr(sA + a * kMmaATile), b0 = smem_addr(sB + b * mma_b_tile(NCOL));
            if (elect_one()) {
#pragma unroll
                for (uint32_t q = 0; q < kMmaK / 16; ++q)
                    mma_bf16(tmem + r * NCOL, mma_sdesc(a0 + 32u * q), mma_sdesc(b0 + 32u * q), idesc, q > 0 ? 1u : 0u);
                mma_commit(&S.sfree[a]);
                mma_commit(&S.bfree[b]);
                mma_commit(&Q.dfull[r]);
            }
            __syncwarp();
            ++issued;
        }
        if (issued > 0 &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(&S.sfree[(issued - 1) % na], ((issued - 1) / na) & 1u)))
            fault = true;
        if ((fault || issued < nk) && lane == 0) {
            atomicOr(p.fault, 4u);
            atomicOr(&s_fault, 1u);
        }
    } else if (warp >= kMgEpiWarp) {
        // rows 32 (warp % 4) + lane: per k-step the region's columns, then
        // y[m] += s[g] * P[g * MP + m] in k order
        const uint32_t row = 32u * (warp & 3u) + lane;
        const uint32_t taddr = tmem + ((32u * (warp & 3u)) << 16);
        for (uint32_t i = 0; i < nk; ++i) {
            const uint32_t a = i % na, ap = (i / na) & 1u, r = i % kMgRegions;
            const bool ok = mbar_wait_bounded(&Q.dfull[r], (i / kMgRegions) & 1u) && mbar_wait_bounded(&S.afull[a], ap);
            if (!__all_sync(0xffffffffu, ok)) {
                fault = true;
                break;
            }
            tc_fence_after();
            uint32_t v[NCU];
            tmem_ldn<NCU>(taddr + r * NCOL, v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&Q.dfree[r]);
            const float* sc = sS + a * (kMmaRows * NG) + row * NG;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const float s = sc[g];
#pragma unroll
                for (int m = 0; m < MP; ++m) y[m] = __fmaf_rn(s, __uint_as_float(v[g * MP + m]), y[m]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&Q.efree[a]);
        }
        if (fault && lane == 0) {
            atomicOr(p.fault, 4u);
            atomicOr(&s_fault, 1u);
        }
    } else {
        const DevTensor& t = p.w;
        const uint32_t r = tid >> 2, quad = tid & 3u;
        const uint64_t n = n0 + r;
        const bool row_ok = n < p.n_rows;
        uint32_t kbi = 0;
        for (uint64_t sp = sp0; sp < sp1 && !fault; ++sp) {
            const uint64_t i = sp - sp0;
            const int s = static_cast<int>(i % p.ns);
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&S.full[s], static_cast<uint32_t>((i / p.ns) & 1u)))) {
                fault = true;
                break;
            }
            const uint64_t k0s = sp * p.span_elems;
            const uint64_t kend = (k0s + p.span_elems < p.K) ? k0s + p.span_elems : p.K;
            const uint8_t* row_in = sP + s * stage_bytes + r * rstride;
            const uint64_t block0 = n * p.bpr + k0s / static_cast<uint64_t>(Fmt<F>::B);
            const uint32_t ph = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(t.x + block0 * Fmt<F>::S) & 15u);
            if constexpr (F == KF_Q6_K) {  // two k-steps at a time from aligned code words
                constexpr int KS = TlQ6K::KS;
                for (uint64_t k0 = k0s; k0 < kend; k0 += KS * kMmaK, kbi += KS) {
                    uint8_t* aS[KS];
                    float* scs[KS];
                    bool ok = true;
#pragma unroll
                    for (int e = 0; e < KS; ++e) {  // the MMAs and the epilogue are done with the stage's previous use
                        const uint32_t kb = kbi + e, a = kb % na;
                        if (kb >= na) {
                            const uint32_t pp = ((kb / na) - 1u) & 1u;
                            ok = ok && mbar_wait_bounded(&S.sfree[a], pp) && mbar_wait_bounded(&Q.efree[a], pp);
                        }
                        aS[e] = sA + a * kMmaATile;
                        scs[e] = sS + a * (kMmaRows * NG);
                    }
                    if (!__all_sync(0xffffffffu, ok)) {
                        fault = true;
                        break;
                    }
                    const uint32_t ks = static_cast<uint32_t>((k0 - k0s) / kMmaK);
                    if (p.aligned)
                        TlQ6K::run<false>(row_in, 0u, ks, quad, aS, scs, r, row_ok);
                    else
                        TlQ6K::run<true>(row_in, ph, ks, quad, aS, scs, r, row_ok);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int e = 0; e < KS; ++e) mbar_arrive(&S.afull[(kbi + e) % na]);
                    }
                }
            } else {
                for (uint64_t k0 = k0s; k0 < kend; k0 += kMmaK, ++kbi) {
                    const uint32_t a = kbi % na;
                    if (kbi >= na) {  // the MMAs and the epilogue are done with this stage's previous use
                        const uint32_t pp = ((kbi / na) - 1u) & 1u;
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait_bounded(&S.sfree[a], pp) && mbar_wait_bounded(&Q.efree[a], pp))) {
                            fault = true;
                            break;
                        }
                    }
                    uint8_t* aS = sA + a * kMmaATile;
                    const uint32_t c = static_cast<uint32_t>((k0 - k0s) / 16u) + quad;
                    const uint64_t kc = k0 + 16u * quad;
                    uint32_t wb[8];
                    float sc = 0.0f;
                    if (row_ok && kc < p.K) {
                        if (p.aligned)
                            Gd::template chunk<false>(row_in, 0u, c, wb, sc);
                        else
                            Gd::template chunk<true>(row_in, ph, c, wb, sc);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) wb[e] = 0u;
                    }
                    *reinterpret_cast<uint4*>(aS + sw128(r, 2u * quad)) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
                    *reinterpret_cast<uint4*>(aS + sw128(r, 2u * quad + 1u)) = make_uint4(wb[4], wb[5], wb[6], wb[7]);
                    if (quad % static_cast<uint32_t>(G / 16) == 0u)
                        sS[a * (kMmaRows * NG) + r * NG + quad / static_cast<uint32_t>(G / 16)] = sc;
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.afull[a]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[s]);
        }
        if (fault && lane == 0) {
            atomicOr(p.fault, 4u);
            atomicOr(&s_fault, 1u);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    fault = s_fault != 0u;

    // y of the epilogue threads: stored, or with split-K parked as
    // part[m * 128 + row] and reduced in rank order (rank r takes rows
    // [r*128/c, (r+1)*128/c) of every activation row)
    const bool split = gridDim.z > 1;
    float* part = reinterpret_cast<float*>(base);
    if (warp >= kMgEpiWarp && warp < kMgEpiWarp + 4) {
        const uint32_t row = 32u * (warp & 3u) + lane;
        const uint64_t nn = n0 + row;
#pragma unroll
        for (int m = 0; m < MP; ++m) {
            const float v = (fault || nk == 0) ? 0.0f : y[m];
            if (split) {
                part[m * kMmaRows + row] = v;
            } else if (!fault && m < p.m_rows && nn < p.n_rows) {
                const uint64_t o = m * p.n_rows + nn;
                if (p.out_bf16)
                    static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(v);
                else
                    static_cast<float*>(p.y)[o] = v;
            }
        }
    }
    if (split) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const uint32_t nr = cluster.num_blocks(), rank = cluster.block_rank();
        const uint32_t rs = kMmaRows * rank / nr, re = kMmaRows * (rank + 1u) / nr;
        for (uint32_t e = tid; e < static_cast<uint32_t>(MP) * (re - rs); e += kMgThreads) {
            const uint32_t m = e / (re - rs), row = rs + e % (re - rs);
            float s = 0.0f;
            for (uint32_t rk = 0; rk < nr; ++rk) {
                const float v = cluster.map_shared_rank(part, rk)[m * kMmaRows + row];
                s = rk == 0 ? v : __fadd_rn(s, v);
            }
            const uint64_t nn = n0 + row;
            if (!fault && m < p.m_rows && nn < p.n_rows) {
                const uint64_t o = m * p.n_rows + nn;
                if (p.out_bf16)
                    static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(s);
                else
                    static_cast<float*>(p.y)[o] = s;
            }
        }
        cluster.sync();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

// Grouped tensor-core kernel of decode family F for MP activation rows (1,
// 2, 4, 8), or nullptr where the family has no grouped codes.
template <int F>
MmaKernelFn mmag_kernel(int mp) {
    if constexpr (Gc<F>::kOk) {
        switch (mp) {
            case 1: return k_mmag<F, 1>;
            case 2: return k_mmag<F, 2>;
            case 4: return k_mmag<F, 4>;
            default: return k_mmag<F, 8>;
        }
    }
    return nullptr;
}

}  // namespace ndq
