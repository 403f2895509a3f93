// Decode kernels specialised for KF_IQ4_NL (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_iq4_nl(int osel) { return kernel_row<KF_IQ4_NL>(osel); }
}  // namespace ndq
