// Decode kernels specialised for gguf:q1_0 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q1_0(int osel) { return kernel_row<KF_Q1_0>(osel); }
}  // namespace ndq
