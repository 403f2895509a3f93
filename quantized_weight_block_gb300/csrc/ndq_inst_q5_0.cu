// Decode kernels specialised for gguf:q5_0 (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_q5_0(int osel) { return kernel_row<KF_Q5_0>(osel); }
MvKernelFn matvec_q5_0(int variant) { return matvec_kernel<KF_Q5_0>(variant); }
MmaKernelFn mma_q5_0() { return mma_kernel<KF_Q5_0>(); }
}  // namespace ndq
