// Decode kernels specialised for KF_NVFP4 (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_nvfp4(int osel) { return kernel_row<KF_NVFP4>(osel); }
MvKernelFn matvec_nvfp4(int variant) { return matvec_kernel<KF_NVFP4>(variant); }
}  // namespace ndq
