// Decode kernels specialised for KF_MXFP4 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_mxfp4(int osel) { return kernel_row<KF_MXFP4>(osel); }
}  // namespace ndq
