// Decode kernels specialised for KF_IQ4_NL (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_iq4_nl(int osel) { return kernel_row<KF_IQ4_NL>(osel); }
MvKernelFn matvec_iq4_nl(int variant) { return matvec_kernel<KF_IQ4_NL>(variant); }
}  // namespace ndq
