// Decode kernels for launches that mix formats: one per output type and one
// that also mixes output types (osel == -1).
#include "ndq_device.cuh"

namespace ndq {
// The generic kernels of each output type sit in their own translation units
// (ndq_inst_generic_<type>.cu) so that they compile in parallel.
KernelFn kernel_generic(int osel) {
    switch (osel) {
        case KO_F32: return kernel_generic_f32();
        case KO_F16: return kernel_generic_f16();
        case KO_BF16: return kernel_generic_bf16();
        case KO_F64: return kernel_generic_f64();
        default: return kernel_generic_any();
    }
}
KernelFn kernel_kquant_mix(int osel) { return kernel_row<kFselKQuantMix>(osel); }

size_t decode_smem_bytes(bool tab, bool lut, bool staged, int stages) {
    return static_cast<size_t>(stages * kInStride + kHdrBytes) + (staged ? kOutStageBytes : 0) +
           (tab ? (lut ? static_cast<size_t>(kLutBytes) : kTabEntries * sizeof(float)) : 0);
}
}  // namespace ndq
