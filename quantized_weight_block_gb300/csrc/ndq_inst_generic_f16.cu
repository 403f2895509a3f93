// Generic (any-format) decode kernel for output type f16.
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_generic_f16() { return k_decode<-1, KO_F16>; }
}  // namespace ndq
