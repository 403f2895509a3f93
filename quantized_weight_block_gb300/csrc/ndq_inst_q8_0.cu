// Decode kernels specialised for KF_Q8_0 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q8_0(int osel) { return kernel_row<KF_Q8_0>(osel); }
}  // namespace ndq
