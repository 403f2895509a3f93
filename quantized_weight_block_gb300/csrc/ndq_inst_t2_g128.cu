// Decode kernels specialised for t2_g128_fp16 (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_t2_g128(int osel) { return kernel_row<KF_T2_G128>(osel); }
MvKernelFn matvec_t2_g128(int variant) { return matvec_kernel<KF_T2_G128>(variant); }
MmaKernelFn mma_t2_g128() { return mma_kernel<KF_T2_G128>(); }
}  // namespace ndq
