// Decode kernels specialised for gguf:q3_k (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_q3_k(int osel) { return kernel_row<KF_Q3_K>(osel); }
}  // namespace ndq
