// Generic (any-format) decode kernel for output type f64.
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_generic_f64() { return k_decode<-1, KO_F64>; }
}  // namespace ndq
