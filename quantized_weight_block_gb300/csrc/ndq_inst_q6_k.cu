// Decode kernels specialised for KF_Q6_K (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q6_k(int osel) { return kernel_row<KF_Q6_K>(osel); }
}  // namespace ndq
