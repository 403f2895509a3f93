// Decode kernels specialised for gguf:iq2_xs (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_iq2_xs(int osel) { return kernel_row<KF_IQ2_XS>(osel); }
MvKernelFn matvec_iq2_xs(int variant) { return matvec_kernel<KF_IQ2_XS>(variant); }
}  // namespace ndq
