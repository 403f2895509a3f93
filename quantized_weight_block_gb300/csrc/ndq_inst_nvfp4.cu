// Decode kernels specialised for KF_NVFP4 (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_nvfp4(int osel) { return kernel_row<KF_NVFP4>(osel); }
MvKernelFn matvec_nvfp4(int variant) { return matvec_kernel<KF_NVFP4>(variant); }
MmaKernelFn mma_nvfp4() { return mma_kernel<KF_NVFP4>(); }
}  // namespace ndq
