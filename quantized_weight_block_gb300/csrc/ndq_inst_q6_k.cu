// Decode kernels specialised for KF_Q6_K (one per output type) and its fused product kernels.
#include "ndq_matvec.cuh"
#include "ndq_mmag.cuh"

namespace ndq {
KernelFn kernel_q6_k(int osel) { return kernel_row<KF_Q6_K>(osel); }
MvKernelFn matvec_q6_k(int variant) { return matvec_kernel<KF_Q6_K>(variant); }
MmaKernelFn mma_q6_k() { return mma_kernel<KF_Q6_K>(); }
MmaKernelFn mmag_q6_k(int mp) { return mmag_kernel<KF_Q6_K>(mp); }
}  // namespace ndq
