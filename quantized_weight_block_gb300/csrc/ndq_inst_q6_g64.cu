// Decode kernels specialised for q6_g64_fp16 (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_q6_g64(int osel) { return kernel_row<KF_Q6_G64>(osel); }
MvKernelFn matvec_q6_g64(int variant) { return matvec_kernel<KF_Q6_G64>(variant); }
MmaKernelFn mma_q6_g64() { return mma_kernel<KF_Q6_G64>(); }
}  // namespace ndq
