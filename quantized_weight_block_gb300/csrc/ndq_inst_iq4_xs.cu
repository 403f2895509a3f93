// Decode kernels specialised for gguf:iq4_xs (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_iq4_xs(int osel) { return kernel_row<KF_IQ4_XS>(osel); }
}  // namespace ndq
