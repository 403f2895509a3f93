// Decode kernels specialised for gguf:iq1_s (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_iq1_s(int osel) { return kernel_row<KF_IQ1_S>(osel); }
MvKernelFn matvec_iq1_s(int variant) { return matvec_kernel<KF_IQ1_S>(variant); }
}  // namespace ndq
