// Decode kernels specialised for gguf:q2_k (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_q2_k(int osel) { return kernel_row<KF_Q2_K>(osel); }
MvKernelFn matvec_q2_k(int variant) { return matvec_kernel<KF_Q2_K>(variant); }
MmaKernelFn mma_q2_k() { return mma_kernel<KF_Q2_K>(); }
}  // namespace ndq
