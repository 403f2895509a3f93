// Decode kernels specialised for gguf:tq1_0 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_tq1_0(int osel) { return kernel_row<KF_TQ1_0>(osel); }
}  // namespace ndq
