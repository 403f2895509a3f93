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
// rows (the MMA's N, 16..256) over all of K, in k-steps of 64:
//   * its 256 threads stage the packed bytes of the tile's rows for a span of
//     max(B, 64) weights (whole blocks) into shared memory, 16-byte lines at a
//     time (every line read holds payload bytes), then decode 64-weight slices
//     of that span with the same Fmt<F> decoders, round them to bfloat16 and
//     write them as the A operand in the 128-byte-swizzled K-major layout;
//   * they copy the X slice [BN x 64] as the B operand in the same layout;
//   * one thread issues four tcgen05.mma (K = 16 each) and commits them to an
//     mbarrier; two operand stages let the next slice be decoded while the
//     tensor core works on the current one;
//   * the epilogue reads the accumulator back with tcgen05.ld (warp w reads
//     TMEM lanes 32*(w%4).., half of the columns each) and stores Y.
// Every wait is bounded; a wait that gives up sets the fault word, and the
// CTA still frees its TMEM before it returns.
#pragma once

#include "ndq_device.cuh"

namespace ndq {
namespace {

constexpr int kMmaThreads = 256;
constexpr int kMmaRows = 128;        // weight rows per CTA (MMA M)
constexpr int kMmaK = 64;            // weights per k-step (one 128-byte swizzle atom of bf16)
constexpr int kMmaATile = kMmaRows * kMmaK * 2;  // 16 KB
constexpr int kMmaStages = 2;

struct MmaShared {
    uint64_t mma_bar[kMmaStages];
    uint32_t tmem;
    uint32_t pad[3];
};

// Dynamic shared memory: [A x2][B x2][packed rows], each 1024-byte aligned.
__host__ __device__ constexpr uint32_t mma_b_tile(uint32_t bn) { return bn * 128u; }
__host__ __device__ constexpr uint32_t mma_row_stride(uint32_t span) { return (span + 15u + 15u + 16u) & ~15u; }
__host__ __device__ constexpr uint32_t mma_smem_bytes(uint32_t bn, uint32_t span) {
    return 1024u + kMmaStages * kMmaATile + kMmaStages * mma_b_tile(bn) +
           ((kMmaRows * mma_row_stride(span) + 1023u) & ~1023u) + 1024u;
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

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <int F>
__global__ void __launch_bounds__(kMmaThreads, 1) k_mma(const MmaParams p) {
    using Fm = Fmt<F>;
    constexpr int CE = Fm::CE;
    extern __shared__ __align__(1024) uint8_t mma_smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mma_smem_raw) + 1023u) & ~uintptr_t(1023));
    const uint32_t bn = static_cast<uint32_t>(p.bn);
    uint8_t* sA = base;
    uint8_t* sB = base + kMmaStages * kMmaATile;
    uint8_t* sP = sB + kMmaStages * mma_b_tile(bn);
    const uint32_t rstride = mma_row_stride(p.span_bytes);
    MmaShared& S = *reinterpret_cast<MmaShared*>(sP + ((kMmaRows * rstride + 1023u) & ~1023u));
    __shared__ SmemHdr H;  // the decoders' 16-entry tables

    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
    const uint32_t ncols = bn < 32u ? 32u : bn;  // TMEM columns (a power of two)
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&S.tmem)),
                     "r"(ncols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int s = 0; s < kMmaStages; ++s) mbar_init(&S.mma_bar[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < 16) {
        H.lut_iq4[tid] = static_cast<float>(c_iq4[tid]);
        H.lut_v[tid] = static_cast<float>(c_v[tid]);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;

    const DevTensor& t = p.w;
    const uint64_t n0 = static_cast<uint64_t>(blockIdx.x) * kMmaRows;
    const uint64_t m0 = static_cast<uint64_t>(blockIdx.y) * bn;
    const uint32_t r = tid & (kMmaRows - 1);  // this thread's weight row in the tile
    const uint32_t half = tid >> 7;           // which half of the row's chunks it decodes
    const uint64_t n = n0 + r;
    const bool row_ok = n < p.n_rows;
    const uint64_t kspan = static_cast<uint64_t>(p.span_elems);  // weights per staged span (whole blocks)
    const uint64_t ksteps = (p.K + kMmaK - 1) / kMmaK;
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((bn >> 3) << 17) | ((kMmaRows >> 4) << 24);
    Ctx x{&H, nullptr, t.divs, 0, t.blocks_per_div, p.grids, code_count(t), n, 0};
    uint32_t phase_row = 0;  // byte phase of this row's staged span
    bool fault = false;

    for (uint64_t kb = 0; kb < ksteps && !fault; ++kb) {
        const int s = static_cast<int>(kb & 1u);
        const uint64_t k0 = kb * kMmaK;
        bool ok = true;
        if (kb >= kMmaStages)  // the MMAs that read stage s two steps ago are done
            ok = mbar_wait_bounded(&S.mma_bar[s], static_cast<uint32_t>(((kb - kMmaStages) >> 1) & 1u));
        if (__syncthreads_or(!ok)) {  // every thread leaves together
            fault = true;
            break;
        }
        if (k0 % kspan == 0) {  // stage the packed span [k0, k0 + kspan) of every row
            __syncthreads();    // every thread is done decoding the previous span
            const uint64_t kleft = p.K - k0;
            const uint64_t blocks = (kleft < kspan ? kleft : kspan) / t.B;  // whole blocks (K % B == 0)
            if (row_ok) {
                const uint8_t* src = t.x + (n * p.bpr + k0 / t.B) * t.S;
                const uint32_t ph = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
                const uint32_t lines = (ph + static_cast<uint32_t>(blocks * t.S) + 15u) >> 4;
                const uint4* gl = reinterpret_cast<const uint4*>(src - ph);
                uint4* sl = reinterpret_cast<uint4*>(sP + r * rstride);
                for (uint32_t i = half; i < lines; i += 2) sl[i] = __ldg(gl + i);
                phase_row = ph;
            }
            x.block0 = n * p.bpr + k0 / t.B;
            x.col0 = k0;
            __syncthreads();
        }
        // decode this k-step's 64 weights of row r into A[s] (bf16, swizzled)
        uint8_t* aS = sA + s * kMmaATile;
        const uint32_t c_first = static_cast<uint32_t>((k0 % kspan) / CE);
        constexpr uint32_t kChunks = kMmaK / CE;        // 4 (CE = 16) or 8 (CE = 8)
        for (uint32_t j = half; j < kChunks; j += 2) {
            const uint64_t kc = k0 + static_cast<uint64_t>(j) * CE;
            uint32_t wb[CE / 2];
            if (row_ok && kc < p.K) {
                float v[CE];
                Fm::template chunk<true>(sP + r * rstride, phase_row, c_first + j, v, x);
#pragma unroll
                for (int i = 0; i < CE / 2; ++i) wb[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
            } else {
#pragma unroll
                for (int i = 0; i < CE / 2; ++i) wb[i] = 0u;
            }
#pragma unroll
            for (int q = 0; q < CE / 8; ++q)
                *reinterpret_cast<uint4*>(aS + sw128(r, j * (CE / 8) + q)) =
                    make_uint4(wb[4 * q], wb[4 * q + 1], wb[4 * q + 2], wb[4 * q + 3]);
        }
        // the activation slice X[m0 .. m0+bn, k0 .. k0+64] into B[s]
        uint8_t* bS = sB + s * mma_b_tile(bn);
        for (uint32_t i = tid; i < bn * 8u; i += kMmaThreads) {
            const uint32_t rr = i >> 3, u = i & 7u;
            const uint64_t m = m0 + rr, kk = k0 + 8u * u;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (m < p.m_rows && kk < p.K) v = __ldg(reinterpret_cast<const uint4*>(p.x + m * p.K + kk));
            *reinterpret_cast<uint4*>(bS + sw128(rr, u)) = v;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t a0 = smem_addr(aS), b0 = smem_addr(bS);
#pragma unroll
            for (uint32_t q = 0; q < kMmaK / 16; ++q)
                mma_bf16(tmem, mma_sdesc(a0 + 32u * q), mma_sdesc(b0 + 32u * q), idesc, (kb > 0 || q > 0) ? 1u : 0u);
            mma_commit(&S.mma_bar[s]);
        }
    }
    // the last commit covers every MMA of the CTA
    if (!fault && ksteps > 0) {
        const uint64_t kl = ksteps - 1;
        const bool ok = mbar_wait_bounded(&S.mma_bar[kl & 1u], static_cast<uint32_t>((kl >> 1) & 1u));
        fault = __syncthreads_or(!ok) != 0;
    }
    tc_fence_after();
    if (fault) {
        if (lane == 0) atomicOr(p.fault, 4u);
    } else {
        // epilogue: warp w reads TMEM lanes 32*(w%4).. (weight rows), columns
        // [half*bn/2, (half+1)*bn/2) (activation rows)
        const uint32_t quarter = warp & 3u, wh = warp >> 2;
        const uint64_t nn = n0 + 32u * quarter + lane;
        const uint32_t cbeg = wh * (bn / 2u), cend = cbeg + bn / 2u;
        for (uint32_t c0 = cbeg; c0 < cend; c0 += 8) {
            uint32_t v[8];
            const uint32_t taddr = tmem + ((32u * quarter) << 16) + c0;
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (nn < p.n_rows) {
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
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols));
}

}  // namespace

// Tensor-core kernel of decode family F (used by the per-format instantiation files).
template <int F>
MmaKernelFn mma_kernel() { return k_mma<F>; }

}  // namespace ndq
