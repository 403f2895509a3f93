// Decode kernels specialised for gguf:iq2_s (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_iq2_s(int osel) { return kernel_row<KF_IQ2_S>(osel); }
MvKernelFn matvec_iq2_s(int variant) { return matvec_kernel<KF_IQ2_S>(variant); }
MmaKernelFn mma_iq2_s() { return mma_kernel<KF_IQ2_S>(); }
}  // namespace ndq
