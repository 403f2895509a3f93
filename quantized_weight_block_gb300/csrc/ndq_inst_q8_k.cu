// Decode kernels specialised for gguf:q8_k (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q8_k(int osel) { return kernel_row<KF_Q8_K>(osel); }
}  // namespace ndq
