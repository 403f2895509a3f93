// Decode kernels specialised for gguf:q5_k (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q5_k(int osel) { return kernel_row<KF_Q5_K>(osel); }
}  // namespace ndq
