// Decode kernels specialised for fp8_e4m3fn_row_fp16 (one per output type).
#include "ndq_device.cuh"

namespace ndq {
KernelFn kernel_fp8_row_fp16(int osel) { return kernel_row<KF_FP8_ROW_FP16>(osel); }
}  // namespace ndq
