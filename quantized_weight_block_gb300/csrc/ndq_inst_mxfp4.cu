// Decode kernels specialised for KF_MXFP4 (one per output type) and its fused product kernel.
#include "ndq_matvec.cuh"

namespace ndq {
KernelFn kernel_mxfp4(int osel) { return kernel_row<KF_MXFP4>(osel); }
MvKernelFn matvec_mxfp4(int variant) { return matvec_kernel<KF_MXFP4>(variant); }
}  // namespace ndq
