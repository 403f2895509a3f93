// Decode kernels specialised for gguf:q2_k (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q2_k(int osel) { return kernel_row<KF_Q2_K>(osel); }
}  // namespace ndq
