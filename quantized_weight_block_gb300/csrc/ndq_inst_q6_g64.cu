// Decode kernels specialised for q6_g64_fp16 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q6_g64(int osel) { return kernel_row<KF_Q6_G64>(osel); }
}  // namespace ndq
