// Decode kernels specialised for q5_g64_fp16 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q5_g64(int osel) { return kernel_row<KF_Q5_G64>(osel); }
}  // namespace ndq
