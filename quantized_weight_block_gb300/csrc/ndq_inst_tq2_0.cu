// Decode kernels specialised for gguf:tq2_0 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_tq2_0(int osel) { return kernel_row<KF_TQ2_0>(osel); }
}  // namespace ndq
