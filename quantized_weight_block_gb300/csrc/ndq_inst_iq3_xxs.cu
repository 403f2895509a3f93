// Decode kernels specialised for gguf:iq3_xxs (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_iq3_xxs(int osel) { return kernel_row<KF_IQ3_XXS>(osel); }
}  // namespace ndq
