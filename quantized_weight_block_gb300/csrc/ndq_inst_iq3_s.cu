// Decode kernels specialised for gguf:iq3_s (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_iq3_s(int osel) { return kernel_row<KF_IQ3_S>(osel); }
}  // namespace ndq
