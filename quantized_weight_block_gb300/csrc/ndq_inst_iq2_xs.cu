// Decode kernels specialised for gguf:iq2_xs (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_iq2_xs(int osel) { return kernel_row<KF_IQ2_XS>(osel); }
}  // namespace ndq
