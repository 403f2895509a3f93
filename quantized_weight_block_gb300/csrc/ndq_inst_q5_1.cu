// Decode kernels specialised for gguf:q5_1 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q5_1(int osel) { return kernel_row<KF_Q5_1>(osel); }
}  // namespace ndq
