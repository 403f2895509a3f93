// Decode kernels specialised for gguf:iq4_xs (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_iq4_xs(int osel) { return kernel_row<KF_IQ4_XS>(osel); }
MvKernelFn matvec_iq4_xs(int variant) { return matvec_kernel<KF_IQ4_XS>(variant); }
MmaKernelFn mma_iq4_xs() { return mma_kernel<KF_IQ4_XS>(); }
}  // namespace ndq
