// Decode kernels specialised for gguf:iq2_s (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_iq2_s(int osel) { return kernel_row<KF_IQ2_S>(osel); }
}  // namespace ndq
