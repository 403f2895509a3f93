// Decode kernels specialised for gguf:tq2_0 (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_tq2_0(int osel) { return kernel_row<KF_TQ2_0>(osel); }
MvKernelFn matvec_tq2_0(int variant) { return matvec_kernel<KF_TQ2_0>(variant); }
MmaKernelFn mma_tq2_0() { return mma_kernel<KF_TQ2_0>(); }
}  // namespace ndq
