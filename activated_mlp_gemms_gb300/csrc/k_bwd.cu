// Backward-pass kernel instances with an MN-major B operand: the dgated /
// dact kernels (dout x Wd with Wd read N-contiguous) and the dx GEMM
// ([dG|dU] x [Wg;Wu] with the weights read N-contiguous).
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_DGATED, false, true, 1>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGATED, false, true, 1>();
template cudaError_t launch_gemm<EPI_DGATED, false, true, 2>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGATED, false, true, 2>();
template cudaError_t launch_gemm<EPI_DACT, false, true, 1>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT, false, true, 1>();
template cudaError_t launch_gemm<EPI_DACT, false, true, 2>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT, false, true, 2>();
template cudaError_t launch_gemm<EPI_STORE_BF16, false, true, 1>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16, false, true, 1>();
template cudaError_t launch_gemm<EPI_STORE_BF16, false, true, 2>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16, false, true, 2>();
}  // namespace mlpk
