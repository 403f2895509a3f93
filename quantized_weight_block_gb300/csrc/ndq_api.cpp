// ndq_api.cpp -- the C ABI declared in include/ndq.h: format registry, host
// validation under the DequantizePacked length rule, and launches.
//
// Validation follows the ONNX "DequantizePacked decoding specification",
// sections "Format identifiers" (closed, case-sensitive identifiers) and
// "Signature and storage" (len(x) == prod(shape[:-1]) * (shape[-1]/B) * S,
// shape[-1] % B == 0, rank >= 1, nonnegative dims, zero dims give empty
// outputs); the nvfp4 divisor words follow NInfer tensor-formats section 3.3
// (one FP32 divisor per stacked source matrix, covering N / D rows).

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <vector>

#include "ndq.h"
#include "ndq_fused.h"
#include "ndq_internal.h"

static_assert(NDQ_NOALLOC_MAX_TENSORS == ndq::kNoAllocMaxTensors, "no-allocation table size");

namespace {

struct FormatRow {
    const char* name;
    int B;
    int S;
    int kfmt;  // ndq::KFmt, or -1 when this build has no decoder
};

// "Quantization formats" table (order = NDQ_GGUF_* ids), then the NInfer
// formats.
const FormatRow kFormats[NDQ_NUM_FORMATS] = {
    {"gguf:q4_0", 32, 18, ndq::KF_Q4_0},
    {"gguf:q4_1", 32, 20, ndq::KF_Q4_1},
    {"gguf:q5_0", 32, 22, ndq::KF_Q5_0},
    {"gguf:q5_1", 32, 24, ndq::KF_Q5_1},
    {"gguf:q8_0", 32, 34, ndq::KF_Q8_0},
    {"gguf:q8_1", 32, 36, ndq::KF_Q8_1},
    {"gguf:q2_k", 256, 84, ndq::KF_Q2_K},
    {"gguf:q3_k", 256, 110, ndq::KF_Q3_K},
    {"gguf:q4_k", 256, 144, ndq::KF_Q4_K},
    {"gguf:q5_k", 256, 176, ndq::KF_Q5_K},
    {"gguf:q6_k", 256, 210, ndq::KF_Q6_K},
    {"gguf:q8_k", 256, 292, ndq::KF_Q8_K},
    {"gguf:iq2_xxs", 256, 66, ndq::KF_IQ2_XXS},
    {"gguf:iq2_xs", 256, 74, ndq::KF_IQ2_XS},
    {"gguf:iq3_xxs", 256, 98, ndq::KF_IQ3_XXS},
    {"gguf:iq1_s", 256, 50, ndq::KF_IQ1_S},
    {"gguf:iq4_nl", 32, 18, ndq::KF_IQ4_NL},
    {"gguf:iq3_s", 256, 110, ndq::KF_IQ3_S},
    {"gguf:iq2_s", 256, 82, ndq::KF_IQ2_S},
    {"gguf:iq4_xs", 256, 136, ndq::KF_IQ4_XS},
    {"gguf:iq1_m", 256, 56, ndq::KF_IQ1_M},
    {"gguf:tq1_0", 256, 54, ndq::KF_TQ1_0},
    {"gguf:tq2_0", 256, 66, ndq::KF_TQ2_0},
    {"gguf:mxfp4", 32, 17, ndq::KF_MXFP4},
    {"gguf:nvfp4", 64, 36, ndq::KF_GGUF_NVFP4},
    {"gguf:q1_0", 128, 18, ndq::KF_Q1_0},
    {"gguf:q2_0", 64, 18, ndq::KF_Q2_0},
    {"nvfp4", 64, 36, ndq::KF_NVFP4},
    {"q4_g64_fp16", 64, 34, ndq::KF_Q4_G64},
    {"q8_g32_fp16", 32, 34, ndq::KF_Q8_0},
    {"q2_g64_fp16", 64, 18, ndq::KF_Q2_0},
    {"q5_g64_fp16", 64, 42, ndq::KF_Q5_G64},
    {"q6_g64_fp16", 64, 50, ndq::KF_Q6_G64},
    {"t2_g128_fp16", 128, 34, ndq::KF_T2_G128},
    {"fp8_e4m3fn_row_bf16", 1, 1, ndq::KF_FP8_ROW_BF16},
    {"fp8_e4m3fn_row_fp16", 1, 1, ndq::KF_FP8_ROW_FP16},
};

bool valid_id(int id) { return id >= 0 && id < NDQ_NUM_FORMATS; }

bool fp8_row(int id) { return id == NDQ_FP8_E4M3FN_ROW_BF16 || id == NDQ_FP8_E4M3FN_ROW_FP16; }

int out_code(int out_dtype, int* size) {
    switch (out_dtype) {
        case NDQ_FLOAT: *size = 4; return ndq::KO_F32;
        case NDQ_FLOAT16: *size = 2; return ndq::KO_F16;
        case NDQ_BFLOAT16: *size = 2; return ndq::KO_BF16;
        case NDQ_DOUBLE: *size = 8; return ndq::KO_F64;
        default: return -1;
    }
}

bool mul_ovf(uint64_t a, uint64_t b, uint64_t* r) { return __builtin_mul_overflow(a, b, r); }

struct Geometry {
    uint64_t nblocks = 0;
    uint64_t nelements = 0;
    uint64_t rows = 0;
    uint64_t ndiv = 0;
};

int geometry(int id, const int64_t* shape, int ndim, uint64_t x_len, Geometry* g) {
    if (!valid_id(id)) return NDQ_ERR_UNKNOWN_FORMAT;
    if (ndim < 1 || ndim > NDQ_MAX_RANK) return NDQ_ERR_BAD_RANK;
    if (!shape) return NDQ_ERR_NULL;
    for (int i = 0; i < ndim; ++i)
        if (shape[i] < 0) return NDQ_ERR_NEGATIVE_DIM;
    const uint64_t B = static_cast<uint64_t>(kFormats[id].B), S = static_cast<uint64_t>(kFormats[id].S);
    const uint64_t K = static_cast<uint64_t>(shape[ndim - 1]);
    if (K % B != 0) return NDQ_ERR_NOT_BLOCK_ALIGNED;
    uint64_t N = 1;
    for (int i = 0; i < ndim - 1; ++i)
        if (mul_ovf(N, static_cast<uint64_t>(shape[i]), &N)) return NDQ_ERR_OVERFLOW;
    uint64_t nb = 0, bytes = 0, elems = 0, out8 = 0;
    if (mul_ovf(N, K / B, &nb) || mul_ovf(nb, S, &bytes) || mul_ovf(N, K, &elems) || mul_ovf(elems, 8, &out8))
        return NDQ_ERR_OVERFLOW;
    if (bytes > static_cast<uint64_t>(INT64_MAX) || out8 > static_cast<uint64_t>(INT64_MAX)) return NDQ_ERR_OVERFLOW;
    uint64_t D = 0;
    if (id == NDQ_NVFP4 && nb > 0) {
        if (x_len < bytes || (x_len - bytes) % 4 != 0) return NDQ_ERR_LENGTH_MISMATCH;
        D = (x_len - bytes) / 4;
        if (D < 1 || N % D != 0) return NDQ_ERR_LENGTH_MISMATCH;
    } else if (fp8_row(id) && nb > 0) {
        // the code plane, then one 16-bit multiplier per row
        if (x_len != bytes + 2u * N) return NDQ_ERR_LENGTH_MISMATCH;
        D = N;
    } else if (x_len != bytes) {
        return NDQ_ERR_LENGTH_MISMATCH;
    }
    g->nblocks = nb;
    g->nelements = elems;
    g->rows = N;
    g->ndiv = D;
    return NDQ_OK;
}

// Full validation of one tensor and its kernel descriptor (tile_begin unset).
int prepare(int id, const int64_t* shape, int ndim, int out_dtype, const uint8_t* x, uint64_t x_len, void* y,
            ndq::DevTensor* t, Geometry* g) {
    if (!valid_id(id)) return NDQ_ERR_UNKNOWN_FORMAT;
    int osize = 0;
    const int oc = out_code(out_dtype, &osize);
    int rc = geometry(id, shape, ndim, x_len, g);
    if (rc != NDQ_OK) return rc;
    if (kFormats[id].kfmt < 0) return NDQ_ERR_UNSUPPORTED_FORMAT;
    if (oc < 0) return NDQ_ERR_BAD_DTYPE;
    if (g->nblocks == 0) return NDQ_OK;
    if (!x || !y) return NDQ_ERR_NULL;
    std::memset(t, 0, sizeof(*t));
    t->x = x;
    t->y = y;
    t->nblocks = g->nblocks;
    t->fmt = kFormats[id].kfmt;
    t->out = oc;
    t->S = static_cast<uint16_t>(kFormats[id].S);
    t->B = static_cast<uint16_t>(kFormats[id].B);
    t->bpt = static_cast<uint16_t>(ndq::kTileElems / kFormats[id].B);
    t->yvec = (reinterpret_cast<uintptr_t>(y) & 15u) == 0;
    if (id == NDQ_NVFP4) {
        const uint64_t bpr = static_cast<uint64_t>(shape[ndim - 1]) / 64u;
        t->divs = x + g->nblocks * 36u;
        t->blocks_per_div = bpr * (g->rows / g->ndiv);
    }
    if (fp8_row(id)) {
        // The kernel reads the code plane in 16-code units (the last one may
        // be partial); the row multipliers follow the codes.
        t->nblocks = (g->nelements + 15u) / 16u;
        t->S = 16;
        t->B = 16;
        t->bpt = static_cast<uint16_t>(ndq::kTileElems / 16);
        t->divs = x + g->nelements;
        t->blocks_per_div = static_cast<uint64_t>(shape[ndim - 1]);
    }
    return NDQ_OK;
}

uint64_t tiles_of(const ndq::DevTensor& t) { return (t.nblocks + t.bpt - 1) / t.bpt; }

constexpr size_t kWorkspaceAlign = 16;

// Activation rows from which bfloat16-weight products run on the tensor cores.
constexpr int64_t kTensorCoreMinRows = 6;

}  // namespace

extern "C" {

int ndq_format_from_name(const char* id) {
    if (!id) return -1;
    for (int i = 0; i < NDQ_NUM_FORMATS; ++i)
        if (std::strcmp(kFormats[i].name, id) == 0) return i;
    return -1;
}

const char* ndq_format_name(int format_id) { return valid_id(format_id) ? kFormats[format_id].name : nullptr; }

int ndq_format_geometry(int format_id, int* B, int* S) {
    if (!valid_id(format_id)) return NDQ_ERR_UNKNOWN_FORMAT;
    if (!B || !S) return NDQ_ERR_NULL;
    *B = kFormats[format_id].B;
    *S = kFormats[format_id].S;
    return NDQ_OK;
}

int ndq_format_supported(int format_id) {
    if (!valid_id(format_id)) return -1;
    return kFormats[format_id].kfmt >= 0 ? 1 : 0;
}

const char* ndq_status_string(int status) {
    switch (status) {
        case NDQ_OK: return "ok";
        case NDQ_ERR_NULL: return "null pointer";
        case NDQ_ERR_UNKNOWN_FORMAT: return "unknown format";
        case NDQ_ERR_UNSUPPORTED_FORMAT: return "format not supported by this build";
        case NDQ_ERR_BAD_RANK: return "bad rank";
        case NDQ_ERR_NEGATIVE_DIM: return "negative dimension";
        case NDQ_ERR_NOT_BLOCK_ALIGNED: return "last dimension not a multiple of the block size";
        case NDQ_ERR_LENGTH_MISMATCH: return "payload length does not match shape";
        case NDQ_ERR_OVERFLOW: return "element or byte count overflows";
        case NDQ_ERR_BAD_DTYPE: return "unsupported output dtype";
        case NDQ_ERR_WORKSPACE: return "workspace missing or too small";
        case NDQ_ERR_CUDA: return "CUDA error";
        case NDQ_ERR_DEVICE_FAULT: return "device fault (bounded wait expired)";
        case NDQ_ERR_BAD_COUNT: return "bad tensor count";
        case NDQ_ERR_TOO_MANY_TENSORS: return "more tensors than the no-allocation launch table holds";
        default: return "unknown status";
    }
}

int ndq_payload_geometry(int format_id, const int64_t* shape, int ndim, uint64_t x_len, uint64_t* nblocks,
                         uint64_t* nelements, uint64_t* ndivisors) {
    Geometry g;
    const int rc = geometry(format_id, shape, ndim, x_len, &g);
    if (rc != NDQ_OK) return rc;
    if (nblocks) *nblocks = g.nblocks;
    if (nelements) *nelements = g.nelements;
    if (ndivisors) *ndivisors = g.ndiv;
    return NDQ_OK;
}

int ndq_dequantize_packed(int format_id, const int64_t* shape, int ndim, int out_dtype, const uint8_t* x_u8,
                          size_t x_len, void* y, void* stream) {
    ndq::KParams p;
    std::memset(&p, 0, sizeof(p));
    Geometry g;
    const int rc = prepare(format_id, shape, ndim, out_dtype, x_u8, x_len, y, &p.single, &g);
    if (rc != NDQ_OK) return rc;
    if (g.nblocks == 0) return NDQ_OK;
    p.single.tile_begin = 0;
    p.table = nullptr;
    p.n = 1;
    p.nv_index = p.single.fmt == ndq::KF_NVFP4 ? 0 : -1;
    p.fsel = p.single.fmt;
    p.osel = p.single.out;
    p.total_tiles = tiles_of(p.single);
    return ndq::launch_decode(p, stream) == 0 ? NDQ_OK : NDQ_ERR_CUDA;
}

// Weights per staged span of the tensor-core products: whole blocks, at
// least 64 (one k-step) and at most 256, as many as keep the span within
// one payload tensor copy (221 bytes: the box of at most 256 bytes also
// holds the line phase and the decoders' over-read).  Fewer, larger copies
// keep more k-steps staged ahead: q8_0 went from 64 to 128 weights per span
// and its [128256,4096] product at M = 8 from 474 to 404 us.
static uint32_t tc_span_elems(uint32_t B, uint32_t S) {
    uint32_t span = B > 64u ? B : 64u;
    while (span * 2u <= 256u && span * 2u / B * S <= 221u) span *= 2u;
    return span;
}

int ndq_matmul_packed(int format_id, int64_t N, int64_t K, const uint8_t* w, size_t w_len, const void* x_bf16,
                      int64_t M, int weight_dtype, int out_dtype, void* y, void* stream) {
    if (!valid_id(format_id)) return NDQ_ERR_UNKNOWN_FORMAT;
    if (N < 0 || K < 0 || M < 0) return NDQ_ERR_NEGATIVE_DIM;
    if (out_dtype != NDQ_FLOAT && out_dtype != NDQ_BFLOAT16) return NDQ_ERR_BAD_DTYPE;
    if (weight_dtype != NDQ_FLOAT && weight_dtype != NDQ_BFLOAT16) return NDQ_ERR_BAD_DTYPE;
    // the fp8 row formats decode in 16-code units, which must not cross rows here
    if (fp8_row(format_id) && K % 16 != 0) return NDQ_ERR_NOT_BLOCK_ALIGNED;
    const int64_t shape[2] = {N, K};
    ndq::MvParams p;
    std::memset(&p, 0, sizeof(p));
    Geometry g;
    // (the weight descriptor's output pointer is unused by the fused kernel)
    const int rc = prepare(format_id, shape, 2, NDQ_FLOAT, w, w_len, const_cast<uint8_t*>(w), &p.w, &g);
    if (rc != NDQ_OK) return rc;
    uint64_t mn = 0, ybytes = 0;
    const uint64_t osize = out_dtype == NDQ_FLOAT ? 4u : 2u;
    if (mul_ovf(static_cast<uint64_t>(M), static_cast<uint64_t>(N), &mn) || mul_ovf(mn, osize, &ybytes) ||
        ybytes > static_cast<uint64_t>(INT64_MAX))
        return NDQ_ERR_OVERFLOW;
    if (mn == 0) return NDQ_OK;
    if (!y || (K > 0 && !x_bf16)) return NDQ_ERR_NULL;
    if (K == 0)  // empty sums
        return cudaMemsetAsync(y, 0, ybytes, static_cast<cudaStream_t>(stream)) == cudaSuccess ? NDQ_OK : NDQ_ERR_CUDA;
    p.n_rows = static_cast<uint64_t>(N);
    p.K = static_cast<uint64_t>(K);
    p.bpr = p.w.nblocks / static_cast<uint64_t>(N);
    const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
    p.xvec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0 && K % 8 == 0;
    p.wbf16 = weight_dtype == NDQ_BFLOAT16;
    // whole rows per staged unit: up to 8192 decoded elements and 8 row groups
    p.rows_per_stage = 1;
    while (p.rows_per_stage < ndq::kConsumerWarpsPerCta &&
           static_cast<int64_t>(p.rows_per_stage) * 2 * K <= ndq::kTileElems)
        p.rows_per_stage *= 2;
    p.out_bf16 = out_dtype == NDQ_BFLOAT16;
    // Six or more activation rows with bfloat16 weights: the tensor-core
    // (tcgen05) product (measured faster than the CUDA-core passes from M = 6
    // on), when X is 16-byte aligned and K % 8 == 0.
    if (weight_dtype == NDQ_BFLOAT16 && M >= kTensorCoreMinRows && p.xvec &&
        (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
        static_cast<uint64_t>(M) <= UINT32_MAX) {
        ndq::MmaParams q;
        std::memset(&q, 0, sizeof(q));
        q.w = p.w;
        q.x = x;
        q.y = y;
        q.n_rows = p.n_rows;
        q.K = p.K;
        q.bpr = p.bpr;
        q.m_rows = static_cast<uint64_t>(M);
        q.bn = 16;
        while (q.bn < 256 && q.bn < static_cast<uint64_t>(M)) q.bn *= 2;
        q.span_elems = tc_span_elems(p.w.B, p.w.S);
        q.span_bytes = q.span_elems / p.w.B * p.w.S;
        q.out_bf16 = p.out_bf16;
        return ndq::launch_mma(q, stream) == 0 ? NDQ_OK : NDQ_ERR_CUDA;
    }
    // Up to 8 activation rows of gguf q8_0 / q4_k / q6_k with K a multiple
    // of 512 and 16-byte-aligned rows, X as binary32 fitting shared memory
    // beside the weight slots (bfloat16 weights: up to 5 rows; one row only
    // for K > 4096): the lean CUDA-core kernel (k_gemvm; X in shared memory,
    // each weight decoded once for all the rows)
    if (M >= 1 && M <= ndq::kMvMaxRows) {
        p.x = x;
        p.y = y;
        p.m = static_cast<int32_t>(M);
        if (ndq::gemvm_takes(p)) return ndq::launch_gemvm(p, stream) == 0 ? NDQ_OK : NDQ_ERR_CUDA;
    }
    // 2 to 8 activation rows with binary32 weights of gguf:q6_k or q8_0 (a
    // group scale times a small code): the grouped tensor-core product (the
    // tensor core sums codes times X per group, the epilogue applies the
    // scales), when X is 16-byte aligned.  (One row stays on the CUDA cores,
    // which measured faster there.)
    if (weight_dtype == NDQ_FLOAT && M >= 2 && M <= ndq::kMvMaxRows && p.xvec && ndq::mmag_for(p.w.fmt, 1) != nullptr) {
        ndq::MmaParams q;
        std::memset(&q, 0, sizeof(q));
        q.w = p.w;
        q.x = x;
        q.y = y;
        q.n_rows = p.n_rows;
        q.K = p.K;
        q.bpr = p.bpr;
        q.m_rows = static_cast<uint64_t>(M);
        q.bn = 1;
        while (q.bn < static_cast<uint64_t>(M)) q.bn *= 2;
        q.span_elems = tc_span_elems(p.w.B, p.w.S);
        q.span_bytes = q.span_elems / p.w.B * p.w.S;
        q.out_bf16 = p.out_bf16;
        return ndq::launch_mmag(q, stream) == 0 ? NDQ_OK : NDQ_ERR_CUDA;
    }
    for (int64_t m0 = 0; m0 < M; m0 += ndq::kMvMaxRows) {
        p.x = x + static_cast<uint64_t>(m0) * static_cast<uint64_t>(K);
        p.y = static_cast<uint8_t*>(y) + static_cast<uint64_t>(m0) * static_cast<uint64_t>(N) * osize;
        p.m = static_cast<int32_t>(M - m0 < ndq::kMvMaxRows ? M - m0 : ndq::kMvMaxRows);
        p.nt = 1;
        p.gt[0].x = p.w.x;
        p.gt[0].y = p.y;
        p.gt[0].rows = p.n_rows;
        if (ndq::launch_matvec(p, stream) != 0) return NDQ_ERR_CUDA;
    }
    return NDQ_OK;
}

int ndq_matmul_packed_batched(const ndq_matmul_desc* descs, int count, int64_t K, const void* x_bf16, int64_t M,
                              int weight_dtype, int out_dtype, void* stream) {
    if (count < 0) return NDQ_ERR_BAD_COUNT;
    if (count == 0) return NDQ_OK;
    if (!descs) return NDQ_ERR_NULL;
    if (K < 0 || M < 0) return NDQ_ERR_NEGATIVE_DIM;
    if (out_dtype != NDQ_FLOAT && out_dtype != NDQ_BFLOAT16) return NDQ_ERR_BAD_DTYPE;
    if (weight_dtype != NDQ_FLOAT && weight_dtype != NDQ_BFLOAT16) return NDQ_ERR_BAD_DTYPE;
    // every product is checked before anything is launched
    ndq::MvParams p;
    std::memset(&p, 0, sizeof(p));
    uint64_t total_rows = 0;
    // (one row with K > 4096 takes k_gemvm in a single call; the batch then
    // runs those calls, so that every output keeps the single call's bits)
    bool one_launch = M == 1 && count <= ndq::kGlMaxTensors && K > 0 && K <= 4096 && x_bf16 != nullptr;
    for (int i = 0; i < count; ++i) {
        const ndq_matmul_desc& d = descs[i];
        if (!valid_id(d.format_id)) return NDQ_ERR_UNKNOWN_FORMAT;
        if (d.n < 0) return NDQ_ERR_NEGATIVE_DIM;
        if (fp8_row(d.format_id) && K % 16 != 0) return NDQ_ERR_NOT_BLOCK_ALIGNED;
        const int64_t shape[2] = {d.n, K};
        ndq::DevTensor t;
        Geometry g;
        const int rc = prepare(d.format_id, shape, 2, NDQ_FLOAT, d.w, d.w_len, const_cast<uint8_t*>(d.w), &t, &g);
        if (rc != NDQ_OK) return rc;
        uint64_t mn = 0, ybytes = 0;
        if (mul_ovf(static_cast<uint64_t>(M), static_cast<uint64_t>(d.n), &mn) ||
            mul_ovf(mn, out_dtype == NDQ_FLOAT ? 4u : 2u, &ybytes) || ybytes > static_cast<uint64_t>(INT64_MAX))
            return NDQ_ERR_OVERFLOW;
        if (mn != 0 && (!d.y || (K > 0 && !x_bf16))) return NDQ_ERR_NULL;
        if (i == 0) p.w = t;
        one_launch = one_launch && d.n > 0 && t.fmt == p.w.fmt;
        if (i < ndq::kGlMaxTensors) {
            p.gt[i].x = d.w;
            p.gt[i].y = d.y;
            p.gt[i].rows = static_cast<uint64_t>(d.n);
        }
        total_rows += static_cast<uint64_t>(d.n);
    }
    if (one_launch) {  // one k_gemvl launch over all the products, when the lean kernel takes them
        p.n_rows = total_rows;
        p.K = static_cast<uint64_t>(K);
        p.bpr = p.w.nblocks / (p.gt[0].rows > 0 ? p.gt[0].rows : 1u);
        p.x = static_cast<const uint16_t*>(x_bf16);
        p.y = descs[0].y;
        p.m = 1;
        p.xvec = (reinterpret_cast<uintptr_t>(x_bf16) & 15u) == 0 && K % 8 == 0;
        p.wbf16 = weight_dtype == NDQ_BFLOAT16;
        p.out_bf16 = out_dtype == NDQ_BFLOAT16;
        p.rows_per_stage = 1;
        p.nt = count;
        if (ndq::gemvl_takes(p)) return ndq::launch_matvec(p, stream) == 0 ? NDQ_OK : NDQ_ERR_CUDA;
    }
    for (int i = 0; i < count; ++i) {
        const ndq_matmul_desc& d = descs[i];
        const int rc = ndq_matmul_packed(d.format_id, d.n, K, d.w, d.w_len, x_bf16, M, weight_dtype, out_dtype, d.y,
                                         stream);
        if (rc != NDQ_OK) return rc;
    }
    return NDQ_OK;
}

size_t ndq_batched_workspace_bytes(int n) {
    if (n < 0) return 0;
    return (static_cast<size_t>(n) * sizeof(ndq::DevTensor) + kWorkspaceAlign - 1) / kWorkspaceAlign *
           kWorkspaceAlign;
}

int ndq_dequantize_packed_batched(const ndq_tensor_desc* descs, int n, void* workspace, size_t ws_bytes,
                                  void* stream) {
    if (n < 0) return NDQ_ERR_BAD_COUNT;
    if (n == 0) return NDQ_OK;
    if (!descs) return NDQ_ERR_NULL;
    std::vector<ndq::DevTensor> table;
    table.reserve(static_cast<size_t>(n));
    uint64_t tiles = 0;
    int nv_index = -1;
    for (int i = 0; i < n; ++i) {
        const ndq_tensor_desc& d = descs[i];
        ndq::DevTensor t;
        Geometry g;
        const int rc = prepare(d.format_id, d.shape, d.ndim, d.out_dtype, d.x, d.x_len, d.y, &t, &g);
        if (rc != NDQ_OK) return rc;
        if (g.nblocks == 0) continue;
        t.tile_begin = tiles;
        tiles += tiles_of(t);
        if (nv_index < 0 && t.fmt == ndq::KF_NVFP4) nv_index = static_cast<int>(table.size());
        table.push_back(t);
    }
    if (table.empty()) return NDQ_OK;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWorkspaceAlign) != 0 ||
        ws_bytes < table.size() * sizeof(ndq::DevTensor))
        return NDQ_ERR_WORKSPACE;
    ndq::DevTensor* dev_table = static_cast<ndq::DevTensor*>(workspace);
    if (ndq::upload_table(dev_table, table.data(), static_cast<int>(table.size()), stream) != 0) return NDQ_ERR_CUDA;
    ndq::KParams p;
    std::memset(&p, 0, sizeof(p));
    p.table = dev_table;
    p.n = static_cast<int32_t>(table.size());
    p.nv_index = nv_index;
    p.total_tiles = tiles;
    ndq::select_kernel(table.data(), static_cast<int>(table.size()), &p.fsel, &p.osel);
    return ndq::launch_decode(p, stream) == 0 ? NDQ_OK : NDQ_ERR_CUDA;
}

int ndq_dequantize_packed_batched_noalloc(const ndq_tensor_desc* descs, int n, void* stream) {
    if (n < 0) return NDQ_ERR_BAD_COUNT;
    if (n > NDQ_NOALLOC_MAX_TENSORS) return NDQ_ERR_TOO_MANY_TENSORS;
    if (n == 0) return NDQ_OK;
    if (!descs) return NDQ_ERR_NULL;
    // Pass 1: validate the whole batch (one bad entry rejects it) and size
    // the launch.  Nothing is kept per tensor, so the host stack holds no
    // table: callers may run on small thread stacks.
    ndq::KernelSelect sel;
    int count = 0;
    uint64_t tiles = 0;
    int nv_index = -1;
    for (int i = 0; i < n; ++i) {
        const ndq_tensor_desc& d = descs[i];
        ndq::DevTensor t;
        Geometry g;
        const int rc = prepare(d.format_id, d.shape, d.ndim, d.out_dtype, d.x, d.x_len, d.y, &t, &g);
        if (rc != NDQ_OK) return rc;
        if (g.nblocks == 0) continue;
        if (nv_index < 0 && t.fmt == ndq::KF_NVFP4) nv_index = count;
        sel.add(t);
        tiles += tiles_of(t);
        ++count;
    }
    if (count == 0) return NDQ_OK;
    ndq::DevTensor* table = nullptr;
    if (ndq::noalloc_table(&table) != 0) return NDQ_ERR_CUDA;
    // Pass 2: the same descriptors again, written into the library's table
    // one upload launch (kUploadChunk entries) at a time.
    ndq::KParams p;
    std::memset(&p, 0, sizeof(p));
    ndq::UploadParams up;
    up.dst = table;
    up.n = 0;
    uint64_t tile_begin = 0;
    int k = 0;
    for (int i = 0; i < n; ++i) {
        const ndq_tensor_desc& d = descs[i];
        ndq::DevTensor t;
        Geometry g;
        if (prepare(d.format_id, d.shape, d.ndim, d.out_dtype, d.x, d.x_len, d.y, &t, &g) != NDQ_OK) return NDQ_ERR_NULL;
        if (g.nblocks == 0) continue;
        t.tile_begin = tile_begin;
        tile_begin += tiles_of(t);
        if (k++ == 0) p.single = t;
        up.d[up.n++] = t;
        if (up.n == ndq::kUploadChunk) {
            if (ndq::upload_chunk(up, stream) != 0) return NDQ_ERR_CUDA;
            up.dst += up.n;
            up.n = 0;
        }
    }
    if (up.n > 0 && ndq::upload_chunk(up, stream) != 0) return NDQ_ERR_CUDA;
    p.table = table;
    p.n = count;
    p.nv_index = nv_index;
    p.total_tiles = tiles;
    sel.get(&p.fsel, &p.osel);
    return ndq::launch_decode(p, stream) == 0 ? NDQ_OK : NDQ_ERR_CUDA;
}

int ndq_test_withhold_copy(int64_t tile, uint32_t wait_limit_us) {
    if (tile < -1 || wait_limit_us == 0 || wait_limit_us > 2000000u) return NDQ_ERR_BAD_COUNT;
    ndq::set_withhold_next(tile, static_cast<uint64_t>(wait_limit_us) * 1000u);
    return NDQ_OK;
}

int ndq_get_device_fault(uint32_t* flags) {
    if (!flags) return NDQ_ERR_NULL;
    return ndq::read_fault(flags) == 0 ? NDQ_OK : NDQ_ERR_CUDA;
}

}  // extern "C"
