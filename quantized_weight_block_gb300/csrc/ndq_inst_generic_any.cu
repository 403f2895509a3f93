// Generic (any-format) decode kernel for mixed output types.
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_generic_any() { return k_decode<-1, -1>; }
}  // namespace ndq
