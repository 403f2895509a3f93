// Decode kernels specialised for gguf:iq2_xxs (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_iq2_xxs(int osel) { return kernel_row<KF_IQ2_XXS>(osel); }
}  // namespace ndq
