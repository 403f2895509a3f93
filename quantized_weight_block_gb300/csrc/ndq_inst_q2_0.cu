// Decode kernels specialised for gguf:q2_0 (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_q2_0(int osel) { return kernel_row<KF_Q2_0>(osel); }
MvKernelFn matvec_q2_0(int variant) { return matvec_kernel<KF_Q2_0>(variant); }
}  // namespace ndq
