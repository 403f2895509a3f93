// Decode kernels specialised for gguf:iq1_s (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_iq1_s(int osel) { return kernel_row<KF_IQ1_S>(osel); }
MvKernelFn matvec_iq1_s(int variant) { return matvec_kernel<KF_IQ1_S>(variant); }
MmaKernelFn mma_iq1_s() { return mma_kernel<KF_IQ1_S>(); }
}  // namespace ndq
