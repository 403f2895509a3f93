// ndq_mma.cuh -- decode fused into a matrix product on the 5th-generation
// tensor cores (tcgen05): the many-activation-row regime (prefill).
//
//     Y[m, n] = sum_k X[m, k] * W[n, k]
//
// W is the payload decoded exactly as DequantizePacked does and rounded once
// to bfloat16 (the tensor-core operand type); X is bfloat16; the tensor core
// accumulates in binary32 in TMEM.
//
// One CTA computes a tile of 128 weight rows (the MMA's M) by BN activation
// rows (the MMA's N, 16..256) over its share of K, in k-steps of 64, with
// warp-specialised roles joined only by mbarriers:
//   * warp 16 (payload producer) stages, for each span of whole blocks (64
//     to 256 weights), the packed bytes of the tile's 128 rows into a ring
//     of up to 4 span stages: one 2-D tensor copy per span from a byte
//     tensor map of the payload when the rows are 16-byte aligned, else
//     asynchronous 16-byte copies of each row's lines (each lane's copies are
//     counted on the span's full barrier as they land);
//   * warps 0-15 (decoders, four threads per weight row) decode each k-step's
//     64 weights of the 128 rows with the Fmt<F> decoders, round them to
//     bfloat16 and write them as the A operand of one of NA operand stages
//     (128-byte-swizzled K-major), then arrive on that stage's A-full
//     barrier;
//   * warp 18 loads the X slice [BN x 64] of each k-step into the stage's B
//     operand with one TMA tensor copy (the 128-byte swizzle is the operand
//     layout; rows and columns outside X read as zero) once the MMAs that
//     last read the stage are done;
//   * warp 17 issues the four tcgen05.mma (K = 16 each) of a k-step once its
//     A and B are full, committing them to the stage's free barrier, which
//     the decoders and the X copies wait on before reusing the stage;
//   * after the k-loop, warps 0-7 read the accumulator back with tcgen05.ld
//     (warp w reads TMEM lanes 32*(w%4).., half of the columns each).  With
//     split-K (gridDim.z > 1, one thread-block cluster per tile) each CTA
//     parks its partial tile in shared memory and rank r adds its share of
//     the columns over every rank's partial in rank order through
//     distributed shared memory, so the result does not depend on timing.
// Every wait is bounded; a wait that gives up sets the fault word and its
// role stops, so every other role's waits run out in turn; every CTA still
// reaches the cluster barriers and frees its TMEM.
#pragma once

#include <cooperative_groups.h>

#include "ndq_device.cuh"
#include "ndq_fused.h"

namespace ndq {
namespace cg = cooperative_groups;
namespace {

constexpr int kMmaDecoders = 512;                     // 16 decode warps
constexpr int kMmaConsumers = 256;                    // the epilogue: warps 0-7
constexpr int kMmaProducerWarp = kMmaDecoders / 32;   // warp 16 stages the payload
constexpr int kMmaIssueWarp = kMmaProducerWarp + 1;   // warp 17 issues the MMAs
constexpr int kMmaXWarp = kMmaProducerWarp + 2;       // warp 18 loads the X slices
constexpr int kMmaThreads = kMmaDecoders + 96;
constexpr int kMmaRows = 128;                         // weight rows per CTA (MMA M)
constexpr int kMmaK = 64;                             // weights per k-step (one 128-byte swizzle atom of bf16)
constexpr int kMmaATile = kMmaRows * kMmaK * 2;       // 16 KB
constexpr uint32_t kMmaMaxStages = 4;                 // A operand stages at most
constexpr uint32_t kMmaMaxB = 8;                      // B operand stages (X slices) at most
constexpr uint32_t kMmaMaxSpans = 4;                  // staged packed spans at most
constexpr uint32_t kMaxMmaSplit = 8;                  // CTAs of a split-K cluster (portable cluster size)
constexpr uint32_t kMmaSmemLimit = 223u * 1024u;      // dynamic shared memory of one CTA at most (227 KB less the static part)

struct MmaShared {
    uint64_t full[kMmaMaxSpans];     // packed span staged (bulk copies complete)
    uint64_t empty[kMmaMaxSpans];    // every decode warp is done with the span
    uint64_t afull[kMmaMaxStages];   // the decode warps wrote the stage's A operand
    uint64_t sfree[kMmaMaxStages];   // the MMAs reading the A stage are done (tcgen05.commit)
    uint64_t bfull[kMmaMaxB];        // the B stage's X slice landed
    uint64_t bfree[kMmaMaxB];        // the MMAs reading the B stage are done (tcgen05.commit)
    uint32_t tmem;
    uint32_t pad[3];
};

// Dynamic shared memory: [A x na][B x nb][packed spans x ns][MmaShared],
// 1024-byte aligned pieces.  After the k-loop the A and B region holds the
// partial tile (128 x bn binary32) of a split-K reduction.
__host__ __device__ constexpr uint32_t mma_b_tile(uint32_t bn) { return bn * 128u; }
// Staged row stride: room for the span, its byte phase and the decoders'
// over-read, rounded to an odd number of 16-byte units so that the rows a
// warp decodes at once spread over the shared-memory banks.
__host__ __device__ constexpr uint32_t mma_row_stride(uint32_t span) {
    return (((span + 15u + 15u + 16u) & ~15u) / 16u % 2u == 0u) ? ((span + 15u + 15u + 16u) & ~15u) + 16u
                                                               : ((span + 15u + 15u + 16u) & ~15u);
}
__host__ __device__ constexpr uint32_t mma_span_stage(uint32_t span) {
    return (kMmaRows * mma_row_stride(span) + 1023u) & ~1023u;
}
// Row bytes of a payload tensor copy: the span from the 16-byte line below
// its first byte plus the decoders' over-read, an odd number of 16-byte
// units (for the banks), at most 256 (a tensor copy's box); 0 if it does
// not fit.  It never exceeds mma_row_stride(span).
__host__ __device__ constexpr uint32_t mma_wbox_odd(uint32_t w) { return (w / 16u) % 2u == 1u ? w : w + 16u; }
__host__ __device__ constexpr uint32_t mma_wbox(uint32_t span) {
    return mma_wbox_odd((span + 20u + 15u) / 16u * 16u) <= 256u ? mma_wbox_odd((span + 20u + 15u) / 16u * 16u) : 0u;
}
__host__ __device__ constexpr uint32_t mma_smem_bytes(uint32_t bn, uint32_t span, uint32_t na, uint32_t ns,
                                                      uint32_t nb) {
    return 1024u + na * kMmaATile + nb * mma_b_tile(bn) + ns * mma_span_stage(span) + 1024u;
}
// A stages na, span stages ns and B stages nb: the deepest A and span
// pipeline that fits with at least na B stages (4, 3, then 2 of each at
// least), then as many B stages as fit, up to 8: the X slices come from L2
// and a deep B ring keeps their latency off the MMA issue.
__host__ __device__ inline void mma_stages(uint32_t bn, uint32_t span, uint32_t* na, uint32_t* ns, uint32_t* nb) {
    *na = 2u;
    *ns = 2u;
    for (uint32_t a = 4u; a >= 2u; --a)
        for (uint32_t s = 4u; s >= 2u; --s)
            if (mma_smem_bytes(bn, span, a, s, a) <= kMmaSmemLimit && a * 8u + s > *na * 8u + *ns &&
                (a >= 3u || s <= 3u)) {
                *na = a;
                *ns = s;
            }
    *nb = *na;
    while (*nb < kMmaMaxB && mma_smem_bytes(bn, span, *na, *ns, *nb + 1u) <= kMmaSmemLimit) ++*nb;
}

// TMA tile copy of a 2-D tensor-map box at (x, y) into shared memory,
// completing its bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// K-major 128-byte swizzle: row r, 16-byte unit u (8 units per 128-byte row).
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t u) {
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((u ^ (r & 7u)) * 16u);
}

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row
// groups 1024 bytes apart.
__device__ __forceinline__ uint64_t mma_sdesc(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;           // leading byte offset (unused for swizzled K-major)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;   // stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;           // fixed 0b001
    d |= static_cast<uint64_t>(2u) << 61;           // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// One lane of the (converged) warp: true in exactly one lane.
__device__ __forceinline__ bool elect_one() {
    uint32_t r;
    asm volatile(
        "{\n.reg .b32 rx;\n.reg .pred px;\n"
        "elect.sync rx|px, 0xffffffff;\nselp.u32 %0, 1, 0, px;\n}\n"
        : "=r"(r));
    return r != 0;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// TMEM -> registers: 8 consecutive binary32 columns of this thread's lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* v) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The span range [sp0, sp1) of packed spans this CTA covers (split-K over
// blockIdx.z).
__device__ __forceinline__ void mma_span_range(const MmaParams& p, uint64_t& sp0, uint64_t& sp1) {
    const uint64_t ns = (p.K + p.span_elems - 1) / p.span_elems;
    sp0 = ns * blockIdx.z / gridDim.z;
    sp1 = ns * (blockIdx.z + 1) / gridDim.z;
}

template <int F>
__device__ void mma_producer(const MmaParams& p, MmaShared& S, uint8_t* sP, uint32_t rstride, uint32_t stage_bytes) {
    constexpr uint32_t B = Fmt<F>::B, SB = Fmt<F>::S;
    const DevTensor& t = p.w;
    const uint32_t lane = threadIdx.x & 31u;
    const int ns = static_cast<int>(p.ns);
    const uint64_t n0 = static_cast<uint64_t>(blockIdx.x) * kMmaRows;
    uint64_t sp0, sp1;
    mma_span_range(p, sp0, sp1);
    int issued = 0;
    bool fault = false;
    if (p.wbox) {  // one tensor copy per span: bytes [x0, x0 + wbox) of the tile's 128 rows, zeros past N
        for (uint64_t sp = sp0; sp < sp1; ++sp, ++issued) {
            const int s = issued % ns;
            if (issued >= ns && !mbar_wait_bounded(&S.empty[s], static_cast<uint32_t>(((issued / ns) - 1) & 1))) {
                fault = true;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&S.full[s], p.wbox * static_cast<uint32_t>(kMmaRows));
                tma_load_2d(sP + s * stage_bytes, &p.wmap, static_cast<int32_t>((sp * p.span_bytes) & ~15ull),
                            static_cast<int32_t>(n0), &S.full[s]);
            }
            __syncwarp();
        }
        if (fault) {
            if (lane == 0) atomicOr(p.fault, 1u);
            for (int j = issued - ns; j < issued; ++j)
                if (j >= 0) mbar_wait_bounded(&S.full[j % ns], static_cast<uint32_t>((j / ns) & 1));
        }
        return;
    }
    for (uint64_t sp = sp0; sp < sp1; ++sp, ++issued) {
        const int s = issued % ns;
        if (issued >= ns && !mbar_wait_bounded(&S.empty[s], static_cast<uint32_t>(((issued / ns) - 1) & 1))) {
            fault = true;
            break;
        }
        const uint64_t k0 = sp * p.span_elems;
        const uint64_t kleft = p.K - k0;
        const uint32_t span = static_cast<uint32_t>((kleft < p.span_elems ? kleft : p.span_elems) / B * SB);
        // every lane copies the 16-byte lines of rows lane, lane + 32, ...
        // (asynchronous copies; the lines all hold payload bytes), then has
        // the full barrier count its arrival once they have landed
        for (uint32_t r = lane; r < kMmaRows; r += 32) {
            const uint64_t n = n0 + r;
            if (n < p.n_rows) {
                const uint8_t* src = t.x + (n * p.bpr + k0 / B) * SB;
                const uint32_t ph = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
                const uint32_t lines = (ph + span + 15u) >> 4;
                const uint8_t* g = src - ph;
                const uint32_t d = smem_addr(sP + s * stage_bytes + r * rstride);
                for (uint32_t i = 0; i < lines; ++i)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + 16u * i), "l"(g + 16u * i)
                                 : "memory");
            }
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(&S.full[s])) : "memory");
    }
    if (fault) {
        if (lane == 0) atomicOr(p.fault, 1u);
        for (int j = issued - ns; j < issued; ++j)
            if (j >= 0) mbar_wait_bounded(&S.full[j % ns], static_cast<uint32_t>((j / ns) & 1));
    }
}

// k-steps of this CTA: K in steps of 64 from its first span (every span but
// a partial last one holds span_elems / 64 k-steps).
__device__ __forceinline__ uint32_t mma_ksteps(const MmaParams& p, uint64_t sp0, uint64_t sp1) {
    const uint64_t k0 = sp0 * p.span_elems;
    const uint64_t k1 = (sp1 * p.span_elems < p.K) ? sp1 * p.span_elems : p.K;
    return static_cast<uint32_t>((k1 - k0 + kMmaK - 1) / kMmaK);
}

template <int F>
__global__ void __launch_bounds__(kMmaThreads, 1) k_mma(const __grid_constant__ MmaParams p) {
    using Fm = Fmt<F>;
    constexpr int CE = Fm::CE;
    extern __shared__ __align__(1024) uint8_t mma_smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mma_smem_raw) + 1023u) & ~uintptr_t(1023));
    const uint32_t bn = p.bn, na = p.na;
    uint8_t* sA = base;
    uint8_t* sB = base + na * kMmaATile;
    uint8_t* sP = sB + na * mma_b_tile(bn);
    const uint32_t rstride = p.wbox ? p.wbox : mma_row_stride(p.span_bytes);
    const uint32_t stage_bytes = mma_span_stage(p.span_bytes);
    MmaShared& S = *reinterpret_cast<MmaShared*>(sP + p.ns * stage_bytes);
    __shared__ SmemHdr H;       // the decoders' 16-entry tables
    __shared__ uint32_t s_fault;  // a role of this CTA gave up a wait

    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
    const uint32_t ncols = bn < 32u ? 32u : bn;  // TMEM columns (a power of two)
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&S.tmem)),
                     "r"(ncols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (uint32_t s = 0; s < p.ns; ++s) {
            mbar_init(&S.full[s], p.wbox ? 1 : 32);  // the tensor copy, or each producer lane's cp.async
            mbar_init(&S.empty[s], kMmaDecoders / 32);
        }
        for (uint32_t s = 0; s < na; ++s) {
            mbar_init(&S.afull[s], kMmaDecoders / 32);
            mbar_init(&S.bfull[s], 1);
            mbar_init(&S.sfree[s], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < 16) {
        H.lut_iq4[tid] = static_cast<float>(c_iq4[tid]);
        H.lut_v[tid] = static_cast<float>(c_v[tid]);
    }
    if (tid == 32) s_fault = 0u;
    if (tid == kMmaXWarp * 32)  // (the X thread) the X map's descriptor into the cache
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.xmap)) : "memory");
    if (tid == kMmaProducerWarp * 32 && p.wbox)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.wmap)) : "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    bool fault = false;
    uint64_t sp0, sp1;
    mma_span_range(p, sp0, sp1);
    const uint32_t nk = mma_ksteps(p, sp0, sp1);
    const uint64_t n0 = static_cast<uint64_t>(blockIdx.x) * kMmaRows;
    const uint64_t m0 = static_cast<uint64_t>(blockIdx.y) * bn;

    if (warp == kMmaProducerWarp) {
        mma_producer<F>(p, S, sP, rstride, stage_bytes);
    } else if (warp == kMmaXWarp) {
        // the X slice of k-step j into stage j % na once the MMAs that read
        // the stage na k-steps ago are done (the whole warp waits, one lane
        // issues the copy)
        const uint32_t xbytes = bn * 128u;
        const uint64_t kx = sp0 * p.span_elems;
        uint32_t b = 0, ph = 0;  // stage and the parity of its previous use
        for (uint32_t j = 0; j < nk; ++j) {
            if (j >= na && !__all_sync(0xffffffffu, mbar_wait_bounded(&S.sfree[b], ph))) {
                if (lane == 0) {
                    atomicOr(p.fault, 4u);
                    atomicOr(&s_fault, 1u);
                }
                break;
            }
            if (elect_one()) {
                mbar_arrive_expect_tx(&S.bfull[b], xbytes);
                tma_load_2d(sB + b * mma_b_tile(bn), &p.xmap, static_cast<int32_t>(kx + static_cast<uint64_t>(kMmaK) * j),
                            static_cast<int32_t>(m0), &S.bfull[b]);
            }
            __syncwarp();
            if (++b == na) {
                b = 0;
                if (j + 1 > na) ph ^= 1u;
            }
        }
    } else if (warp == kMmaIssueWarp) {
        // the MMAs of k-step i once the decoders filled A and the copy filled
        // B; the whole warp waits and computes the descriptors (warp-uniform
        // values), one lane issues
        const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((bn >> 3) << 17) | ((kMmaRows >> 4) << 24);
        uint32_t issued = 0;  // k-steps whose MMAs were issued
        uint32_t a = 0, ph = 0;
        for (uint32_t i = 0; i < nk; ++i) {
            const bool ok = mbar_wait_bounded(&S.afull[a], ph) && mbar_wait_bounded(&S.bfull[a], ph);
            if (!__all_sync(0xffffffffu, ok)) {
                fault = true;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_addr(sA + a * kMmaATile), b0 = smem_addr(sB + a * mma_b_tile(bn));
            if (elect_one()) {
#pragma unroll
                for (uint32_t q = 0; q < kMmaK / 16; ++q)
                    mma_bf16(tmem, mma_sdesc(a0 + 32u * q), mma_sdesc(b0 + 32u * q), idesc, (i > 0 || q > 0) ? 1u : 0u);
                mma_commit(&S.sfree[a]);
            }
            __syncwarp();
            ++issued;
            if (++a == na) {
                a = 0;
                ph ^= 1u;
            }
        }
        // the last commit covers every MMA issued (also after a fault: no
        // MMA may still run when the epilogue reads or frees TMEM)
        if (issued > 0 &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(&S.sfree[(issued - 1) % na], ((issued - 1) / na) & 1u)))
            fault = true;
        if ((fault || issued < nk) && lane == 0) {
            atomicOr(p.fault, 4u);
            atomicOr(&s_fault, 1u);
        }
    } else {
        const DevTensor& t = p.w;
        // four adjacent threads per weight row (a warp touches 8 rows at a
        // time, which spread over the shared-memory banks)
        const uint32_t r = tid >> 2;      // this thread's weight row in the tile
        const uint32_t quad = tid & 3u;   // which quarter of the row's chunks it decodes
        const uint64_t n = n0 + r;
        const bool row_ok = n < p.n_rows;
        Ctx x{&H, nullptr, t.divs, 0, t.blocks_per_div, p.grids, code_count(t), n, 0};
        uint32_t kbi = 0;  // k-steps decoded by this CTA
        uint32_t sa = 0, fph = 1;  // operand stage of k-step kbi, parity of its previous use
        constexpr uint32_t kChunks = kMmaK / CE;
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
            x.block0 = n * p.bpr + k0s / Fm::B;
            const uint32_t ph = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(t.x + x.block0 * Fm::S) & 15u);
            x.col0 = k0s;
            for (uint64_t k0 = k0s; k0 < kend; k0 += kMmaK, ++kbi) {
                const uint32_t a = sa;
                // the MMAs that read this stage na k-steps ago are done (fph:
                // the parity of that use's completion)
                if (kbi >= na && !__all_sync(0xffffffffu, mbar_wait_bounded(&S.sfree[a], fph))) {
                    fault = true;
                    break;
                }
                if (++sa == na) {
                    sa = 0;
                    fph ^= 1u;
                }
                // this k-step's 64 weights of row r into A[a] (bf16, swizzled)
                uint8_t* aS = sA + a * kMmaATile;
                const uint32_t c_first = static_cast<uint32_t>((k0 - k0s) / CE);
                for (uint32_t j = quad; j < kChunks; j += 4) {
                    const uint64_t kc = k0 + static_cast<uint64_t>(j) * CE;
                    uint32_t wb[CE / 2];
                    if (row_ok && kc < p.K) {
                        float v[CE];
                        if (p.aligned)  // (every staged row starts on a 16-byte boundary)
                            Fm::template chunk<false>(row_in, 0u, c_first + j, v, x);
                        else
                            Fm::template chunk<true>(row_in, ph, c_first + j, v, x);
#pragma unroll
                        for (int e = 0; e < CE / 2; ++e) wb[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
                    } else {
#pragma unroll
                        for (int e = 0; e < CE / 2; ++e) wb[e] = 0u;
                    }
#pragma unroll
                    for (int q = 0; q < CE / 8; ++q)
                        *reinterpret_cast<uint4*>(aS + sw128(r, j * (CE / 8) + q)) =
                            make_uint4(wb[4 * q], wb[4 * q + 1], wb[4 * q + 2], wb[4 * q + 3]);
                }
                fence_proxy_async_smem();  // the tensor core reads A through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.afull[a]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[s]);  // this warp no longer reads the span
        }
        if (fault && lane == 0) {
            atomicOr(p.fault, 4u);
            atomicOr(&s_fault, 1u);
        }
    }
    // every role is done: the MMA thread has seen its last commit complete
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool issued_any = nk > 0;
    fault = s_fault != 0u;  // a faulted tile writes zeros (the fault word reports it)

    // Epilogue.  Warp w < 8 reads TMEM lanes 32*(w%4).. (weight rows) and half
    // of the columns (activation rows).  With one CTA per tile it stores Y.
    // With a split-K cluster every CTA parks its partial tile in shared
    // memory, column-major (part[c * 128 + row], so a warp's 32 rows are one
    // conflict-free line), and rank r then reduces columns
    // [r*bn/c, (r+1)*bn/c) of every rank's partial, adding them in rank
    // order so that the result does not depend on timing.
    const bool split = gridDim.z > 1;
    float* part = reinterpret_cast<float*>(base);  // [bn][128] binary32, over the operand stages
    const uint32_t quarter = warp & 3u, wh = (warp >> 2) & 1u;
    const uint32_t row = 32u * quarter + lane;
    const uint32_t cbeg = wh * (bn / 2u), cend = cbeg + bn / 2u;
    if (tid < kMmaConsumers) {
        const uint64_t nn = n0 + row;
        for (uint32_t c0 = cbeg; c0 < cend; c0 += 8) {
            uint32_t v[8];
            tmem_ld8(tmem + ((32u * quarter) << 16) + c0, v);
            if (split) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    part[(c0 + j) * kMmaRows + row] = (fault || !issued_any) ? 0.0f : __uint_as_float(v[j]);
            } else if (!fault && issued_any && nn < p.n_rows) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint64_t m = m0 + c0 + j;
                    if (m < p.m_rows) {
                        const uint64_t o = m * p.n_rows + nn;
                        if (p.out_bf16)
                            static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(__uint_as_float(v[j]));
                        else
                            static_cast<float*>(p.y)[o] = __uint_as_float(v[j]);
                    }
                }
            }
        }
    }
    if (split) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();  // every CTA's partial tile is in its shared memory
        const uint32_t nr = cluster.num_blocks(), rank = cluster.block_rank();
        const uint32_t cs = bn * rank / nr, ce = bn * (rank + 1u) / nr;
        const uint32_t units = (ce - cs) * (kMmaRows / 4u);  // float4 units of this rank's columns
        if (tid < kMmaConsumers) {
            const float4* src[kMaxMmaSplit];
#pragma unroll
            for (uint32_t rk = 0; rk < kMaxMmaSplit; ++rk)
                src[rk] = reinterpret_cast<const float4*>(cluster.map_shared_rank(part, rk < nr ? rk : 0u)) +
                          cs * (kMmaRows / 4u);
            for (uint32_t u = tid; u < units; u += kMmaConsumers) {
                float4 pv[kMaxMmaSplit];
#pragma unroll
                for (uint32_t rk = 0; rk < kMaxMmaSplit; ++rk)
                    if (rk < nr) pv[rk] = src[rk][u];
                float4 s = pv[0];
#pragma unroll
                for (uint32_t rk = 1; rk < kMaxMmaSplit; ++rk)
                    if (rk < nr) {
                        s.x = __fadd_rn(s.x, pv[rk].x);
                        s.y = __fadd_rn(s.y, pv[rk].y);
                        s.z = __fadd_rn(s.z, pv[rk].z);
                        s.w = __fadd_rn(s.w, pv[rk].w);
                    }
                const uint64_t m = m0 + cs + u / (kMmaRows / 4u);
                const uint64_t nb = n0 + 4u * (u % (kMmaRows / 4u));
                const float sv[4] = {s.x, s.y, s.z, s.w};
                if (m < p.m_rows) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (nb + j < p.n_rows) {
                            const uint64_t o = m * p.n_rows + nb + j;
                            if (p.out_bf16)
                                static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(sv[j]);
                            else
                                static_cast<float*>(p.y)[o] = sv[j];
                        }
                }
            }
        }
        cluster.sync();  // every rank has read the partials before any CTA exits
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols));
}

}  // namespace

// Tensor-core kernel of decode family F (used by the per-format instantiation files).
template <int F>
MmaKernelFn mma_kernel() { return k_mma<F>; }

}  // namespace ndq
