// Decode kernels specialised for gguf:q3_k (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_q3_k(int osel) { return kernel_row<KF_Q3_K>(osel); }
MvKernelFn matvec_q3_k(int variant) { return matvec_kernel<KF_Q3_K>(variant); }
MmaKernelFn mma_q3_k() { return mma_kernel<KF_Q3_K>(); }
}  // namespace ndq
