// Decode kernels specialised for fp8_e4m3fn_row_fp16 (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_fp8_row_fp16(int osel) { return kernel_row<KF_FP8_ROW_FP16>(osel); }
MvKernelFn matvec_fp8_row_fp16(int variant) { return matvec_kernel<KF_FP8_ROW_FP16>(variant); }
MmaKernelFn mma_fp8_row_fp16() { return mma_kernel<KF_FP8_ROW_FP16>(); }
}  // namespace ndq
