// Launcher of the fused decode + product kernels (one per decode family,
// instantiated beside each family's decode kernels).
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "ndq_matvec.cuh"
#include "ndq_mmag.cuh"

namespace ndq {

MvKernelFn matvec_for(int kfmt, int variant) {
    switch (kfmt) {
        case KF_FP8_ROW_BF16: return matvec_fp8_row_bf16(variant);
        case KF_FP8_ROW_FP16: return matvec_fp8_row_fp16(variant);
        case KF_GGUF_NVFP4: return matvec_gguf_nvfp4(variant);
        case KF_IQ1_M: return matvec_iq1_m(variant);
        case KF_IQ1_S: return matvec_iq1_s(variant);
        case KF_IQ2_S: return matvec_iq2_s(variant);
        case KF_IQ2_XS: return matvec_iq2_xs(variant);
        case KF_IQ2_XXS: return matvec_iq2_xxs(variant);
        case KF_IQ3_S: return matvec_iq3_s(variant);
        case KF_IQ3_XXS: return matvec_iq3_xxs(variant);
        case KF_IQ4_NL: return matvec_iq4_nl(variant);
        case KF_IQ4_XS: return matvec_iq4_xs(variant);
        case KF_MXFP4: return matvec_mxfp4(variant);
        case KF_NVFP4: return matvec_nvfp4(variant);
        case KF_Q1_0: return matvec_q1_0(variant);
        case KF_Q2_0: return matvec_q2_0(variant);
        case KF_Q2_K: return matvec_q2_k(variant);
        case KF_Q3_K: return matvec_q3_k(variant);
        case KF_Q4_0: return matvec_q4_0(variant);
        case KF_Q4_1: return matvec_q4_1(variant);
        case KF_Q4_G64: return matvec_q4_g64(variant);
        case KF_Q4_K: return matvec_q4_k(variant);
        case KF_Q5_0: return matvec_q5_0(variant);
        case KF_Q5_1: return matvec_q5_1(variant);
        case KF_Q5_G64: return matvec_q5_g64(variant);
        case KF_Q5_K: return matvec_q5_k(variant);
        case KF_Q6_G64: return matvec_q6_g64(variant);
        case KF_Q6_K: return matvec_q6_k(variant);
        case KF_Q8_0: return matvec_q8_0(variant);
        case KF_Q8_1: return matvec_q8_1(variant);
        case KF_Q8_K: return matvec_q8_k(variant);
        case KF_T2_G128: return matvec_t2_g128(variant);
        case KF_TQ1_0: return matvec_tq1_0(variant);
        case KF_TQ2_0: return matvec_tq2_0(variant);
        default: return nullptr;
    }
}

namespace {
constexpr int kMvSmemBuckets = static_cast<int>(kMvXBytes / 8192) + 1;  // activation copies in 8 KB steps
struct MvDeviceInfo {
    int sms = 0;
    bool attr_set[KF_COUNT][kMvVariants] = {};
    int ctas_per_sm[KF_COUNT][kMvVariants][kMvSmemBuckets] = {};  // 0 = not yet queried
    int lean_slot[KF_COUNT][kMvVariants] = {};  // the lean kernel: slot of the last query and its result
    int lean_cps[KF_COUNT][kMvVariants] = {};
};
MvDeviceInfo g_mv_dev[64];
}  // namespace

bool gemvl_takes(const MvParams& p) {
    const int f = p.w.fmt;
    if (p.m != 1 || p.K == 0 || p.K % kGlIter != 0 || p.K / kGlIter > 4u * kConsumerWarpsPerCta || f < 0 ||
        f >= KF_COUNT || p.nt < 1 || p.nt > kGlMaxTensors || (p.bpr * p.w.S) % 16u != 0)
        return false;
    for (int t = 0; t < p.nt; ++t)
        if ((reinterpret_cast<uintptr_t>(p.gt[t].x) & 15u) != 0) return false;
    return matvec_for(f, kMvLean) != nullptr;
}

int launch_matvec(const MvParams& p0, void* stream) {
    if (p0.n_rows == 0 || p0.m <= 0) return 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    MvParams p = p0;
    const int se = device_symbols(dev, &p.fault, &p.grids);
    if (se != 0) return se;
    const int f = p.w.fmt;
    // every unit starts on a 16-byte boundary when the payload does and a
    // unit's rows (or a row, when rows are segmented) span whole lines;
    // segments of a row are whole tiles, which always do
    const uint64_t unit_rows = static_cast<uint64_t>(p.rows_per_stage);
    const bool aligned = (reinterpret_cast<uintptr_t>(p.w.x) & 15u) == 0 && (unit_rows * p.bpr * p.w.S) % 16u == 0;
    // the activations: one row as binary32 or several as bfloat16 in shared
    // memory when they fit, else read from global memory
    const uint64_t xf32 = p.K * 4u, xbf16 = static_cast<uint64_t>(p.m) * p.K * 2u;
    // one row: k_gemv1 (a warp per weight row) when the row fits
    bool rows_aligned = (reinterpret_cast<uintptr_t>(p.w.x) & 15u) == 0 && (p.bpr * p.w.S) % 16u == 0;
    for (int t = 0; t < p.nt; ++t) rows_aligned = rows_aligned && (reinterpret_cast<uintptr_t>(p.gt[t].x) & 15u) == 0;
    int variant = kMvAnyAlign;
    uint64_t xbytes = 0;
    if (p.m == 1 && xf32 <= kMvXBytes) {
        variant = rows_aligned ? kMvOneRowF32 : kMvOneRowF32Any;
        xbytes = xf32;
    } else if (aligned && p.m > 1 && p.xvec && xbf16 <= kMvXBytes) {
        variant = kMvRowsBf16;
        xbytes = xbf16;
    } else if (aligned) {
        variant = kMvRowsGlobal;
    }
    // one row of a K-quant format with whole 512-weight iterations: the lean
    // kernel (activations in registers, CTAs taking row blocks in turn)
    MvKernelFn fn = nullptr;
    const uint64_t nit = p.K / kGlIter;
    if (p.m == 1 && rows_aligned && p.K % kGlIter == 0 && nit <= 4u * kConsumerWarpsPerCta && f >= 0 &&
        f < KF_COUNT) {
        const int xr = nit <= 8u ? 0 : nit <= 16u ? 1 : 2;
        const int lv = kMvLean + 2 * xr + (p.wbf16 ? 1 : 0);
        fn = matvec_for(f, lv);
        if (fn) {
            variant = lv;
            xbytes = 0;
        }
    }
    if (!fn && p.nt > 1) return static_cast<int>(cudaErrorInvalidValue);  // (several tensors: the lean kernel only)
    if (!fn) fn = (f >= 0 && f < KF_COUNT) ? matvec_for(f, variant) : nullptr;
    if (!fn) return static_cast<int>(cudaErrorInvalidDeviceFunction);
    const bool lean = variant >= kMvLean;
    const bool one_row = variant == kMvOneRowF32 || variant == kMvOneRowF32Any;
    MvDeviceInfo& di = g_mv_dev[dev];
    if (di.sms == 0) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return static_cast<int>(e);
        di.sms = sms;
    }
    if (lean) {  // rows per stage (for two resident CTAs per SM) and the slot they take
        const uint32_t xr = static_cast<uint32_t>(1 << ((variant - kMvLean) / 2));
        p.rows_per_stage = static_cast<int32_t>(
            gemvl_rows_per_stage(p.n_rows, p.bpr * p.w.S, xr, 2u * static_cast<uint64_t>(di.sms)));
        p.slot = static_cast<int32_t>(gl_slot_bytes(p.bpr * p.w.S, static_cast<uint32_t>(p.rows_per_stage)));
        if (p.nt < 1 || p.nt > kGlMaxTensors) return static_cast<int>(cudaErrorInvalidValue);
        uint64_t blocks = 0;
        for (int t = 0; t < p.nt; ++t) {
            blocks += (p.gt[t].rows + static_cast<uint64_t>(p.rows_per_stage) - 1) / static_cast<uint64_t>(p.rows_per_stage);
            p.gt[t].blk_end = blocks;
        }
    }
    const size_t base = lean      ? gemvl_smem_bytes(static_cast<uint32_t>(p.slot))
                        : one_row ? gemv1_smem_base(p.w.B, p.w.S)
                                  : static_cast<size_t>(kStages * kInStride + kHdrBytes + kMvExtraBytes);
    const int bucket = static_cast<int>((xbytes + 8191u) / 8192u);
    const size_t smem = base + static_cast<size_t>(bucket) * 8192u;
    if (!di.attr_set[f][variant]) {
        const size_t most = lean ? gemvl_smem_bytes(kGlSlotMax) : base + kMvXBytes;
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(most));
        if (e != cudaSuccess) return static_cast<int>(e);
        di.attr_set[f][variant] = true;
    }
    // (the lean kernel's occupancy depends on its slot size: the last query
    // per kernel is kept)
    if (lean && di.lean_slot[f][variant] != p.slot) {
        di.lean_slot[f][variant] = p.slot;
        di.lean_cps[f][variant] = 0;
    }
    int& cps = lean ? di.lean_cps[f][variant] : di.ctas_per_sm[f][variant][bucket];
    if (cps == 0) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kBlockThreads, smem);
        if (e != cudaSuccess) return static_cast<int>(e);
        cps = n > 0 ? n : 1;
    }
    const uint64_t R = static_cast<uint64_t>(one_row ? kGvRows : p.rows_per_stage);
    // (k_gemv1: blocks of 8 rows; k_gemvl: the row blocks of all its tensors)
    const uint64_t units = lean ? p.gt[p.nt - 1].blk_end : (p.n_rows + R - 1) / R;
    const uint64_t resident = static_cast<uint64_t>(di.sms) * static_cast<uint64_t>(cps);
    const unsigned grid = static_cast<unsigned>(units < resident ? units : resident);
    void* args[] = {&p};
    // programmatic stream serialization: the kernel waits on the previous
    // grid itself (griddepcontrol.wait), after warming L2 with its weights
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kBlockThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(fn), args);
    return static_cast<int>(e);
}

// Activation rows of the k_gemvm kernel for m rows.
static uint32_t gm_mp(int32_t m) { return m <= 1 ? 1u : m <= 2 ? 2u : m <= 4 ? 4u : 8u; }

// Shared memory of a k_gemvm launch with rb rows per stage.
static size_t gm_smem_of(const MvParams& p, uint32_t rb) {
    return gm_smem_bytes(gl_slot_bytes(p.bpr * p.w.S, rb), gm_mp(p.m), p.K, rb);
}

bool gemvm_takes(const MvParams& p) {
    const int f = p.w.fmt;
    if (p.m < 1 || p.m > kMvMaxRows || p.K == 0 || p.K % kGlIter != 0 || p.K > 32u * kGlIter ||
        (p.m == 1 && p.K <= 8u * kGlIter) || f < 0 || f >= KF_COUNT || (p.bpr * p.w.S) % 16u != 0 ||
        (reinterpret_cast<uintptr_t>(p.w.x) & 15u) != 0)
        return false;
    const uint32_t mp = gm_mp(p.m);
    if (gm_smem_of(p, kGmQuad * gm_row_groups(static_cast<uint32_t>(p.K / kGlIter), mp)) > kGmSmemMax) return false;
    return matvec_for(f, kMvMulti) != nullptr;
}

int launch_gemvm(const MvParams& p0, void* stream) {
    if (p0.n_rows == 0) return 0;
    if (!gemvm_takes(p0)) return static_cast<int>(cudaErrorInvalidValue);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    MvParams p = p0;
    const int se = device_symbols(dev, &p.fault, &p.grids);
    if (se != 0) return se;
    const int f = p.w.fmt;
    const uint32_t mp = gm_mp(p.m);
    const bool mi = p.K / kGlIter > gm_warps(mp);
    const int variant =
        kMvMulti + 4 * (mp == 1u ? 0 : mp == 2u ? 1 : mp == 4u ? 2 : 3) + (mi ? 2 : 0) + (p.wbf16 ? 1 : 0);
    const MvKernelFn fn = matvec_for(f, variant);
    if (!fn) return static_cast<int>(cudaErrorInvalidDeviceFunction);
    MvDeviceInfo& di = g_mv_dev[dev];
    if (di.sms == 0) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return static_cast<int>(e);
        di.sms = sms;
    }
    // rows per stage: 4 rg pp (every row group takes pp quads), the most
    // (pp <= 4) that fit one CTA per SM and leave at least two row blocks
    // per CTA
    const uint32_t nit = static_cast<uint32_t>(p.K / kGlIter);
    const uint32_t rg = gm_row_groups(nit, mp);
    const uint64_t rowb = p.bpr * p.w.S;
    const uint64_t sms = static_cast<uint64_t>(di.sms);
    auto smem_of = [&](uint32_t pp) { return gm_smem_of(p, kGmQuad * rg * pp); };
    uint32_t pp = 4;
    while (pp > 1u && (smem_of(pp) > kGmSmemMax ||
                       (p.n_rows + kGmQuad * rg * pp - 1u) / (kGmQuad * rg * pp) < 2u * sms))
        pp >>= 1;
    const size_t smem = smem_of(pp);
    if (smem > kGmSmemMax) return static_cast<int>(cudaErrorInvalidValue);
    const uint32_t rb = kGmQuad * rg * pp;
    p.rows_per_stage = static_cast<int32_t>(rb);
    p.slot = static_cast<int32_t>(gl_slot_bytes(rowb, rb));
    if (!di.attr_set[f][variant]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kGmSmemMax));
        if (e != cudaSuccess) return static_cast<int>(e);
        di.attr_set[f][variant] = true;
    }
    const uint64_t nblk = (p.n_rows + rb - 1u) / rb;
    const unsigned grid = static_cast<unsigned>(nblk < sms ? nblk : sms);
    void* args[] = {&p};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(gm_warps(mp) * 32u);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(fn), args);
    return static_cast<int>(e);
}

MmaKernelFn mma_for(int kfmt) {
    switch (kfmt) {
        case KF_FP8_ROW_BF16: return mma_fp8_row_bf16();
        case KF_FP8_ROW_FP16: return mma_fp8_row_fp16();
        case KF_GGUF_NVFP4: return mma_gguf_nvfp4();
        case KF_IQ1_M: return mma_iq1_m();
        case KF_IQ1_S: return mma_iq1_s();
        case KF_IQ2_S: return mma_iq2_s();
        case KF_IQ2_XS: return mma_iq2_xs();
        case KF_IQ2_XXS: return mma_iq2_xxs();
        case KF_IQ3_S: return mma_iq3_s();
        case KF_IQ3_XXS: return mma_iq3_xxs();
        case KF_IQ4_NL: return mma_iq4_nl();
        case KF_IQ4_XS: return mma_iq4_xs();
        case KF_MXFP4: return mma_mxfp4();
        case KF_NVFP4: return mma_nvfp4();
        case KF_Q1_0: return mma_q1_0();
        case KF_Q2_0: return mma_q2_0();
        case KF_Q2_K: return mma_q2_k();
        case KF_Q3_K: return mma_q3_k();
        case KF_Q4_0: return mma_q4_0();
        case KF_Q4_1: return mma_q4_1();
        case KF_Q4_G64: return mma_q4_g64();
        case KF_Q4_K: return mma_q4_k();
        case KF_Q5_0: return mma_q5_0();
        case KF_Q5_1: return mma_q5_1();
        case KF_Q5_G64: return mma_q5_g64();
        case KF_Q5_K: return mma_q5_k();
        case KF_Q6_G64: return mma_q6_g64();
        case KF_Q6_K: return mma_q6_k();
        case KF_Q8_0: return mma_q8_0();
        case KF_Q8_1: return mma_q8_1();
        case KF_Q8_K: return mma_q8_k();
        case KF_T2_G128: return mma_t2_g128();
        case KF_TQ1_0: return mma_tq1_0();
        case KF_TQ2_0: return mma_tq2_0();
        default: return nullptr;
    }
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;  // (benign race: same value)
    if (!encode) {
        void* fp = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fp) return nullptr;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fp);
    }
    return encode;
}

// The payload as a byte tensor [N, bpr * S] for one tensor copy per staged
// span (rows 16-byte aligned and a span that fits a box); else wbox = 0 and
// the producer copies 16-byte lines.
int payload_map(MmaParams& p) {
    p.wbox = 0;
    const uint64_t row_bytes = p.bpr * p.w.S;
    const uint32_t wbox = mma_wbox(p.span_bytes);
    if (wbox == 0u || (reinterpret_cast<uintptr_t>(p.w.x) & 15u) != 0u || row_bytes % 16u != 0u) return 0;
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return static_cast<int>(cudaErrorNotSupported);
    const cuuint64_t gdim[2] = {row_bytes, p.n_rows};
    const cuuint64_t gstride[1] = {row_bytes};
    const cuuint32_t box[2] = {wbox, static_cast<cuuint32_t>(kMmaRows)};
    const cuuint32_t estride[2] = {1u, 1u};
    if (encode(&p.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.w.x), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return static_cast<int>(cudaErrorInvalidValue);
    p.wbox = wbox;
    return 0;
}
}  // namespace

int launch_mma(const MmaParams& p0, void* stream) {
    if (p0.n_rows == 0 || p0.m_rows == 0) return 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    MmaParams p = p0;
    const int se = device_symbols(dev, &p.fault, &p.grids);
    if (se != 0) return se;
    const int f = p.w.fmt;
    const MmaKernelFn fn = (f >= 0 && f < KF_COUNT) ? mma_for(f) : nullptr;
    if (!fn) return static_cast<int>(cudaErrorInvalidDeviceFunction);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    // (bn: the smallest power of two >= M up to 256, so that each weight is
    // decoded once per 256 activation rows; short grids split K instead)
    // (k_mma's B stages are its A stages: a deeper B ring measured slower)
    mma_stages(p.bn, p.span_bytes, &p.na, &p.ns, &p.nb);
    p.nb = p.na;
    p.aligned = (reinterpret_cast<uintptr_t>(p.w.x) & 15u) == 0 && (p.bpr * p.w.S) % 16u == 0 && p.span_bytes % 16u == 0;
    const size_t smem = mma_smem_bytes(p.bn, p.span_bytes, p.na, p.ns, p.nb);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return static_cast<int>(e);
    // X as a 2-D tensor map: [m_rows, K] bfloat16, boxes of 64 columns (one
    // 128-byte swizzle span) by bn rows, zero outside X
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return static_cast<int>(cudaErrorNotSupported);
    const int pm = payload_map(p);
    if (pm != 0) return pm;
    const cuuint64_t gdim[2] = {p.K, p.m_rows};
    const cuuint64_t gstride[1] = {p.K * 2u};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kMmaK), p.bn};
    const cuuint32_t estride[2] = {1u, 1u};
    if (encode(&p.xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.x), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return static_cast<int>(cudaErrorInvalidValue);
    const uint64_t tiles_n = (p.n_rows + kMmaRows - 1) / kMmaRows;
    const uint64_t tiles_m = (p.m_rows + p.bn - 1) / p.bn;
    // Split K over a thread-block cluster of up to 8 CTAs (each CTA's partial
    // tile, 128 x bn binary32, is parked over its operand and span stages;
    // every CTA keeps at least two spans): the largest split whose CTAs
    // number at most one per SM (one CTA fills an SM's shared memory).
    const uint64_t spans = (p.K + p.span_elems - 1) / p.span_elems;
    const uint64_t tiles = tiles_n * tiles_m;
    const uint64_t max_ctas = static_cast<uint64_t>(sms);
    const bool parks = static_cast<uint64_t>(p.bn) * kMmaRows * 4u <=
                       static_cast<uint64_t>(p.na) * kMmaATile + static_cast<uint64_t>(p.nb) * mma_b_tile(p.bn) +
                           static_cast<uint64_t>(p.ns) * mma_span_stage(p.span_bytes);
    unsigned split = 1;
    while (split < kMaxMmaSplit && parks && spans >= 4u * split && tiles * 2u * split <= max_ctas) split *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles_n), static_cast<unsigned>(tiles_m), split);
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = split;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&p};
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(fn), args);
    return static_cast<int>(e);
}

MmaKernelFn mmag_for(int kfmt, int mp) {
    switch (kfmt) {
        case KF_Q6_K: return mmag_q6_k(mp);
        case KF_Q8_0: return mmag_q8_0(mp);
        default: return nullptr;
    }
}

namespace {
// Weights per scale group of the grouped families (k_mmag).
int mmag_group(int kfmt) { return kfmt == KF_Q6_K ? Gc<KF_Q6_K>::G : Gc<KF_Q8_0>::G; }
}  // namespace

int launch_mmag(const MmaParams& p0, void* stream) {
    if (p0.n_rows == 0 || p0.m_rows == 0) return 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    MmaParams p = p0;
    const int se = device_symbols(dev, &p.fault, &p.grids);
    if (se != 0) return se;
    const int f = p.w.fmt;
    const MmaKernelFn fn = (f >= 0 && f < KF_COUNT) ? mmag_for(f, static_cast<int>(p.bn)) : nullptr;
    if (!fn) return static_cast<int>(cudaErrorInvalidDeviceFunction);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    const int ng = kMmaK / mmag_group(f);
    const uint32_t ncol = mg_ncol(ng, p.bn);
    mmag_stages(ncol, ng, p.span_bytes, &p.na, &p.ns, &p.nb);
    p.aligned = (reinterpret_cast<uintptr_t>(p.w.x) & 15u) == 0 && (p.bpr * p.w.S) % 16u == 0 && p.span_bytes % 16u == 0;
    const int pm = payload_map(p);
    if (pm != 0) return pm;
    const size_t smem = mmag_smem_bytes(ncol, ng, p.span_bytes, p.na, p.ns, p.nb);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return static_cast<int>(e);
    // Split K over a cluster of up to 8 CTAs while the tiles leave SMs idle
    // (every CTA keeps at least four spans; the partial rows, MP x 128
    // binary32, are parked over the operand stages)
    const uint64_t tiles = (p.n_rows + kMmaRows - 1) / kMmaRows;
    const uint64_t spans = (p.K + p.span_elems - 1) / p.span_elems;
    unsigned split = 1;
    while (split < kMaxMmaSplit && spans >= 8u * split && tiles * 2u * split <= static_cast<uint64_t>(sms)) split *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles), 1u, split);
    cfg.blockDim = dim3(kMgThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = split;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void* args[] = {&p};
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(fn), args);
    return static_cast<int>(e);
}

}  // namespace ndq
