// Decode kernels specialised for gguf:iq3_s (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_iq3_s(int osel) { return kernel_row<KF_IQ3_S>(osel); }
MvKernelFn matvec_iq3_s(int variant) { return matvec_kernel<KF_IQ3_S>(variant); }
}  // namespace ndq
