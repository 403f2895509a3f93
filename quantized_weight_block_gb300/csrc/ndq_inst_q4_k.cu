// Decode kernels specialised for KF_Q4_K (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_q4_k(int osel) { return kernel_row<KF_Q4_K>(osel); }
MvKernelFn matvec_q4_k(int variant) { return matvec_kernel<KF_Q4_K>(variant); }
MmaKernelFn mma_q4_k() { return mma_kernel<KF_Q4_K>(); }
}  // namespace ndq
