// Decode kernels specialised for gguf:iq1_s (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_iq1_s(int osel) { return kernel_row<KF_IQ1_S>(osel); }
}  // namespace ndq
