// Decode kernels for launches that mix formats: one per output type and one
// that also mixes output types (osel == -1).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_generic(int osel) { return kernel_row<-1>(osel); }
KernelFn kernel_kquant_mix(int osel) { return kernel_row<kFselKQuantMix>(osel); }

size_t decode_smem_bytes(bool tab) {
    return static_cast<size_t>(kStages * kInStride + kHdrBytes) + (tab ? kTabEntries * sizeof(float) : 0);
}
}  // namespace ndq
