// Decode kernels specialised for gguf:iq1_m (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_iq1_m(int osel) { return kernel_row<KF_IQ1_M>(osel); }
}  // namespace ndq
