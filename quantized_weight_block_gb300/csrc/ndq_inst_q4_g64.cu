// Decode kernels specialised for KF_Q4_G64 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q4_g64(int osel) { return kernel_row<KF_Q4_G64>(osel); }
}  // namespace ndq
