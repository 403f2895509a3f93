// ndq_fused.h -- launch descriptors of the decode fused into a matrix
// product (ndq_matvec.cuh, ndq_mma.cuh, ndq_mmag.cuh), shared by the host
// ABI (ndq_api.cpp) and the launchers (ndq_inst_matvec.cu).  Not part of the
// public ABI.
#pragma once

#include <cuda.h>  // CUtensorMap (the tensor-core products' activation and payload maps)

#include "ndq_internal.h"

namespace ndq {

// Decode fused into a product with few activation rows (ndq_matvec.cuh):
// Y[m, n] = sum_k X[m, k] * W[n, k] for m < m_rows <= kMvMaxRows.
constexpr int kMvMaxRows = 8;
// One weight tensor of a k_gemvl launch: its payload rows, its outputs and
// the end of its row blocks in the launch's block order.
constexpr int kGlMaxTensors = 8;
struct GlTensor {
    const uint8_t* x;  // payload [rows, K] (16-byte-aligned rows)
    void* y;           // outputs [rows] (the launch's output type)
    uint64_t rows;
    uint64_t blk_end;  // (set by the launcher) row blocks of tensors 0..this one
};

struct MvParams {
    DevTensor w;          // the weight payload as a decode descriptor (y unused)
    const uint16_t* x;    // bfloat16 activations [m, K], row-major
    void* y;              // outputs [m, N], row-major (FLOAT or BFLOAT16)
    uint64_t n_rows;      // N
    uint64_t K;
    uint64_t bpr;         // payload blocks per weight row
    int32_t m;            // activation rows of this launch (1..kMvMaxRows)
    int32_t xvec;         // 1 if every 16-element slice of x is 16-byte aligned
    int32_t rows_per_stage;  // R in {1, 2, 4, 8}: whole rows per staged unit (K <= 8192/R), 1 = segments
    int32_t wbf16;        // 1: round the decoded weights to bfloat16 before the product
    int32_t out_bf16;     // 1: y is bfloat16, else binary32
    int32_t slot;         // k_gemvl: bytes of one staged row slot (set by the launcher)
    unsigned int* fault;  // device fault word (set by the launcher)
    const IqGrids* grids;  // IQ codebooks (set by the launcher)
    // k_gemvl: the launch's tensors (same format and K; n_rows is their
    // total); a single product is tensor 0 = (w.x, y, n_rows)
    int32_t nt;
    int32_t pad2_;
    GlTensor gt[kGlMaxTensors];
};

using MvKernelFn = void (*)(MvParams);
// True when the lean one-row kernel (k_gemvl) takes the launch p: one row of
// X, K a multiple of 512 up to 16384, a family with lean decoders, and
// 16-byte-aligned rows in every tensor of p.gt.
bool gemvl_takes(const MvParams& p);

// Where a fused kernel reads the activations: a copy in shared memory
// (binary32 for one row, bfloat16 for several) when it fits in kMvXBytes,
// else global memory.
constexpr uint64_t kMvXBytes = 64 * 1024;
enum MvX : int { kMvXGlobal = 0, kMvXF32 = 1, kMvXBf16 = 2 };
// Fused kernel variants: 16-byte-aligned payload with one activation row in
// shared memory (binary32), several rows in shared memory (bfloat16), several
// rows from global memory; and any payload alignment (rows from global).
enum MvVariant : int {
    kMvOneRowF32 = 0,     // one row (k_gemv1), rows 16-byte aligned
    kMvRowsBf16 = 1,
    kMvRowsGlobal = 2,
    kMvAnyAlign = 3,
    kMvOneRowF32Any = 4,  // one row (k_gemv1), any alignment
    // one row, lean per-format decoders (k_gemvl, gguf q8_0 / q4_k / q6_k):
    // kMvLean + 2 * xr + wbf16, xr = 0, 1, 2 for 1, 2, 4 units per lane
    kMvLean = 5,
    // X in shared memory, lean decoders (k_gemvm): kMvMulti + 4 * mpi +
    // 2 * mi + wbf16, mpi = 0, 1, 2, 3 for kernels of 1, 2, 4, 8 activation
    // rows, mi = 1 when a warp takes several iterations of a row
    kMvMulti = 11,
    kMvVariants = 27
};
// True when the lean kernel with X in shared memory (k_gemvm) takes the
// launch p: 1 <= m <= 8 (m == 1 only for K > 4096, where it measured
// faster than k_gemvl), K a multiple of 512 up to 16384, X as binary32 and
// three slots of 4 rows fitting one CTA's shared memory, a family with lean
// decoders, one tensor (p.w) with 16-byte-aligned rows.
bool gemvm_takes(const MvParams& p);
int launch_gemvm(const MvParams& p, void* stream);

// Decode fused into a tensor-core (tcgen05) product (ndq_mma.cuh): tiles of
// 128 weight rows by bn activation rows, the weights rounded to bfloat16.
struct MmaParams {
    DevTensor w;          // the weight payload as a decode descriptor (y unused)
    const uint16_t* x;    // bfloat16 activations [m_rows, K], 16-byte aligned, K % 8 == 0
    void* y;              // outputs [m_rows, N]
    uint64_t n_rows;      // N
    uint64_t K;
    uint64_t bpr;         // payload blocks per weight row
    uint64_t m_rows;      // M
    uint32_t bn;          // activation rows per CTA: 16, 32, 64, 128 or 256
    uint32_t span_elems;  // weights per staged span: max(B, 64), whole blocks
    uint32_t span_bytes;  // payload bytes of a full span
    int32_t out_bf16;
    uint32_t na;          // operand stages (A and B tiles in flight), 2..4 (set by the launcher)
    uint32_t ns;          // staged payload spans, 2..4 (set by the launcher)
    uint32_t aligned;     // 1: the payload, its rows and its spans start on 16-byte boundaries
    uint32_t wbox;        // bytes per row of a payload tensor copy (wmap), 0: 16-byte copies per row
    uint32_t nb;          // B operand stages (X slices in flight), 2..8 (set by the launcher)
    uint32_t pad_;
    unsigned int* fault;
    const IqGrids* grids;
    CUtensorMap xmap;     // X as a 2-D bfloat16 tensor [m_rows, K], boxes of 64 x bn, 128-byte swizzle
    CUtensorMap wmap;     // (wbox > 0) the payload as bytes [N, bpr * S], boxes of wbox x 128 rows
};
using MmaKernelFn = void (*)(MmaParams);
// The grouped tensor-core product with binary32 weights (k_mmag), for the
// families whose weight is a group scale times a code exact in bfloat16:
// the kernel for mp = 1, 2, 4 or 8 activation rows, or nullptr.
MmaKernelFn mmag_q6_k(int mp);
MmaKernelFn mmag_q8_0(int mp);
MmaKernelFn mmag_for(int kfmt, int mp);
int launch_mmag(const MmaParams& p, void* stream);
MmaKernelFn mma_fp8_row_bf16();
MmaKernelFn mma_fp8_row_fp16();
MmaKernelFn mma_gguf_nvfp4();
MmaKernelFn mma_iq1_m();
MmaKernelFn mma_iq1_s();
MmaKernelFn mma_iq2_s();
MmaKernelFn mma_iq2_xs();
MmaKernelFn mma_iq2_xxs();
MmaKernelFn mma_iq3_s();
MmaKernelFn mma_iq3_xxs();
MmaKernelFn mma_iq4_nl();
MmaKernelFn mma_iq4_xs();
MmaKernelFn mma_mxfp4();
MmaKernelFn mma_nvfp4();
MmaKernelFn mma_q1_0();
MmaKernelFn mma_q2_0();
MmaKernelFn mma_q2_k();
MmaKernelFn mma_q3_k();
MmaKernelFn mma_q4_0();
MmaKernelFn mma_q4_1();
MmaKernelFn mma_q4_g64();
MmaKernelFn mma_q4_k();
MmaKernelFn mma_q5_0();
MmaKernelFn mma_q5_1();
MmaKernelFn mma_q5_g64();
MmaKernelFn mma_q5_k();
MmaKernelFn mma_q6_g64();
MmaKernelFn mma_q6_k();
MmaKernelFn mma_q8_0();
MmaKernelFn mma_q8_1();
MmaKernelFn mma_q8_k();
MmaKernelFn mma_t2_g128();
MmaKernelFn mma_tq1_0();
MmaKernelFn mma_tq2_0();
MmaKernelFn mma_for(int kfmt);
int launch_mma(const MmaParams& p, void* stream);

// Fused kernels, one per decode family (defined in the instantiation files).
MvKernelFn matvec_fp8_row_bf16(int variant);
MvKernelFn matvec_fp8_row_fp16(int variant);
MvKernelFn matvec_gguf_nvfp4(int variant);
MvKernelFn matvec_iq1_m(int variant);
MvKernelFn matvec_iq1_s(int variant);
MvKernelFn matvec_iq2_s(int variant);
MvKernelFn matvec_iq2_xs(int variant);
MvKernelFn matvec_iq2_xxs(int variant);
MvKernelFn matvec_iq3_s(int variant);
MvKernelFn matvec_iq3_xxs(int variant);
MvKernelFn matvec_iq4_nl(int variant);
MvKernelFn matvec_iq4_xs(int variant);
MvKernelFn matvec_mxfp4(int variant);
MvKernelFn matvec_nvfp4(int variant);
MvKernelFn matvec_q1_0(int variant);
MvKernelFn matvec_q2_0(int variant);
MvKernelFn matvec_q2_k(int variant);
MvKernelFn matvec_q3_k(int variant);
MvKernelFn matvec_q4_0(int variant);
MvKernelFn matvec_q4_1(int variant);
MvKernelFn matvec_q4_g64(int variant);
MvKernelFn matvec_q4_k(int variant);
MvKernelFn matvec_q5_0(int variant);
MvKernelFn matvec_q5_1(int variant);
MvKernelFn matvec_q5_g64(int variant);
MvKernelFn matvec_q5_k(int variant);
MvKernelFn matvec_q6_g64(int variant);
MvKernelFn matvec_q6_k(int variant);
MvKernelFn matvec_q8_0(int variant);
MvKernelFn matvec_q8_1(int variant);
MvKernelFn matvec_q8_k(int variant);
MvKernelFn matvec_t2_g128(int variant);
MvKernelFn matvec_tq1_0(int variant);
MvKernelFn matvec_tq2_0(int variant);
MvKernelFn matvec_for(int kfmt, int variant);

// Launch one fused product.  Returns 0 or a CUDA error code.
int launch_matvec(const MvParams& p, void* stream);

}  // namespace ndq
