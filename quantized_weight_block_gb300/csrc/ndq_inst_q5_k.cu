// Decode kernels specialised for gguf:q5_k (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_q5_k(int osel) { return kernel_row<KF_Q5_K>(osel); }
MvKernelFn matvec_q5_k(int variant) { return matvec_kernel<KF_Q5_K>(variant); }
}  // namespace ndq
