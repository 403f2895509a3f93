// Decode kernels specialised for KF_Q4_0 (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_q4_0(int osel) { return kernel_row<KF_Q4_0>(osel); }
MvKernelFn matvec_q4_0(int variant) { return matvec_kernel<KF_Q4_0>(variant); }
}  // namespace ndq
