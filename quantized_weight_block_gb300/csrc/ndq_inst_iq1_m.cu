// Decode kernels specialised for gguf:iq1_m (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_iq1_m(int osel) { return kernel_row<KF_IQ1_M>(osel); }
MvKernelFn matvec_iq1_m(int variant) { return matvec_kernel<KF_IQ1_M>(variant); }
MmaKernelFn mma_iq1_m() { return mma_kernel<KF_IQ1_M>(); }
}  // namespace ndq
