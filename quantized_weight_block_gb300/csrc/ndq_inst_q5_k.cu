// Decode kernels specialised for gguf:q5_k (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_q5_k(int osel) { return kernel_row<KF_Q5_K>(osel); }
MvKernelFn matvec_q5_k(int variant) { return matvec_kernel<KF_Q5_K>(variant); }
MmaKernelFn mma_q5_k() { return mma_kernel<KF_Q5_K>(); }
}  // namespace ndq
