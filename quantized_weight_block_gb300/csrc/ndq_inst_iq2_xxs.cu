// Decode kernels specialised for gguf:iq2_xxs (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_iq2_xxs(int osel) { return kernel_row<KF_IQ2_XXS>(osel); }
MvKernelFn matvec_iq2_xxs(int variant) { return matvec_kernel<KF_IQ2_XXS>(variant); }
}  // namespace ndq
