// Decode kernels specialised for KF_NVFP4 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_nvfp4(int osel) { return kernel_row<KF_NVFP4>(osel); }
}  // namespace ndq
