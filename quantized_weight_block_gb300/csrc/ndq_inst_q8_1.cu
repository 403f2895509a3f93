// Decode kernels specialised for gguf:q8_1 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q8_1(int osel) { return kernel_row<KF_Q8_1>(osel); }
}  // namespace ndq
