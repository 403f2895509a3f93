// Decode kernels specialised for gguf:q4_1 (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_q4_1(int osel) { return kernel_row<KF_Q4_1>(osel); }
MvKernelFn matvec_q4_1(int variant) { return matvec_kernel<KF_Q4_1>(variant); }
MmaKernelFn mma_q4_1() { return mma_kernel<KF_Q4_1>(); }
}  // namespace ndq
