// Decode kernels specialised for gguf:q5_0 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q5_0(int osel) { return kernel_row<KF_Q5_0>(osel); }
}  // namespace ndq
