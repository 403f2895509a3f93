// Decode kernels specialised for gguf:iq2_xxs (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_iq2_xxs(int osel) { return kernel_row<KF_IQ2_XXS>(osel); }
MvKernelFn matvec_iq2_xxs(int variant) { return matvec_kernel<KF_IQ2_XXS>(variant); }
MmaKernelFn mma_iq2_xxs() { return mma_kernel<KF_IQ2_XXS>(); }
}  // namespace ndq
