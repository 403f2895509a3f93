// Decode kernels specialised for KF_Q8_0 (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mmag.cuh"

namespace ndq {
KernelFn kernel_q8_0(int osel) { return kernel_row<KF_Q8_0>(osel); }
MvKernelFn matvec_q8_0(int variant) { return matvec_kernel<KF_Q8_0>(variant); }
MmaKernelFn mma_q8_0() { return mma_kernel<KF_Q8_0>(); }
MmaKernelFn mmag_q8_0(int mp) { return mmag_kernel<KF_Q8_0>(mp); }
}  // namespace ndq
