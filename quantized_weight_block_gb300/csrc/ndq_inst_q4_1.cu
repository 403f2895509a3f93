// Decode kernels specialised for gguf:q4_1 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q4_1(int osel) { return kernel_row<KF_Q4_1>(osel); }
}  // namespace ndq
