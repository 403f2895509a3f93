// Decode kernels specialised for gguf:tq2_0 (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_tq2_0(int osel) { return kernel_row<KF_TQ2_0>(osel); }
MvKernelFn matvec_tq2_0(int variant) { return matvec_kernel<KF_TQ2_0>(variant); }
}  // namespace ndq
