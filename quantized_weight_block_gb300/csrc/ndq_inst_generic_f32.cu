// Generic (any-format) decode kernel for output type f32.
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_generic_f32() { return k_decode<-1, KO_F32>; }
}  // namespace ndq
