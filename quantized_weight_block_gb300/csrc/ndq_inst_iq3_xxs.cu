// Decode kernels specialised for gguf:iq3_xxs (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_iq3_xxs(int osel) { return kernel_row<KF_IQ3_XXS>(osel); }
MvKernelFn matvec_iq3_xxs(int variant) { return matvec_kernel<KF_IQ3_XXS>(variant); }
MmaKernelFn mma_iq3_xxs() { return mma_kernel<KF_IQ3_XXS>(); }
}  // namespace ndq
