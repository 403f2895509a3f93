// Decode kernels specialised for gguf:iq4_xs (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_iq4_xs(int osel) { return kernel_row<KF_IQ4_XS>(osel); }
MvKernelFn matvec_iq4_xs(int variant) { return matvec_kernel<KF_IQ4_XS>(variant); }
}  // namespace ndq
