// Generic (any-format) decode kernel for output type bf16.
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_generic_bf16() { return k_decode<-1, KO_BF16>; }
}  // namespace ndq
