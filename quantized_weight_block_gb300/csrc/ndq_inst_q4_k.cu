// Decode kernels specialised for KF_Q4_K (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q4_k(int osel) { return kernel_row<KF_Q4_K>(osel); }
}  // namespace ndq
