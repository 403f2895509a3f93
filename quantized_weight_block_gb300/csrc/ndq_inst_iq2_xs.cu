// Decode kernels specialised for gguf:iq2_xs (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_iq2_xs(int osel) { return kernel_row<KF_IQ2_XS>(osel); }
MvKernelFn matvec_iq2_xs(int variant) { return matvec_kernel<KF_IQ2_XS>(variant); }
MmaKernelFn mma_iq2_xs() { return mma_kernel<KF_IQ2_XS>(); }
}  // namespace ndq
