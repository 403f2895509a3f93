// Decode kernels specialised for gguf:iq1_m (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_iq1_m(int osel) { return kernel_row<KF_IQ1_M>(osel); }
MvKernelFn matvec_iq1_m(int variant) { return matvec_kernel<KF_IQ1_M>(variant); }
}  // namespace ndq
