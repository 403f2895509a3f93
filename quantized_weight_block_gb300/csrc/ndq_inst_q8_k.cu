// Decode kernels specialised for gguf:q8_k (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_q8_k(int osel) { return kernel_row<KF_Q8_K>(osel); }
MvKernelFn matvec_q8_k(int variant) { return matvec_kernel<KF_Q8_K>(variant); }
MmaKernelFn mma_q8_k() { return mma_kernel<KF_Q8_K>(); }
}  // namespace ndq
