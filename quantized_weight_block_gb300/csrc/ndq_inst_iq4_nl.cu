// Decode kernels specialised for KF_IQ4_NL (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_iq4_nl(int osel) { return kernel_row<KF_IQ4_NL>(osel); }
MvKernelFn matvec_iq4_nl(int variant) { return matvec_kernel<KF_IQ4_NL>(variant); }
MmaKernelFn mma_iq4_nl() { return mma_kernel<KF_IQ4_NL>(); }
}  // namespace ndq
