// Decode kernels specialised for gguf:iq3_s (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_iq3_s(int osel) { return kernel_row<KF_IQ3_S>(osel); }
MvKernelFn matvec_iq3_s(int variant) { return matvec_kernel<KF_IQ3_S>(variant); }
MmaKernelFn mma_iq3_s() { return mma_kernel<KF_IQ3_S>(); }
}  // namespace ndq
