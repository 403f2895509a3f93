// Decode kernels specialised for t2_g128_fp16 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_t2_g128(int osel) { return kernel_row<KF_T2_G128>(osel); }
}  // namespace ndq
