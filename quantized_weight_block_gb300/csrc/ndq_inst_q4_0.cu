// Decode kernels specialised for KF_Q4_0 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q4_0(int osel) { return kernel_row<KF_Q4_0>(osel); }
}  // namespace ndq
