// Decode kernels specialised for KF_MXFP4 (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mma.cuh"

namespace ndq {
KernelFn kernel_mxfp4(int osel) { return kernel_row<KF_MXFP4>(osel); }
MvKernelFn matvec_mxfp4(int variant) { return matvec_kernel<KF_MXFP4>(variant); }
MmaKernelFn mma_mxfp4() { return mma_kernel<KF_MXFP4>(); }
}  // namespace ndq
