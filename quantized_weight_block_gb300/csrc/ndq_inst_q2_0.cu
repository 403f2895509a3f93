// Decode kernels specialised for gguf:q2_0 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q2_0(int osel) { return kernel_row<KF_Q2_0>(osel); }
}  // namespace ndq
