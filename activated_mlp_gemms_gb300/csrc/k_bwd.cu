// Backward-pass kernel instances with an MN-major B operand: the dgated /
// dact kernels (dout x Wd with Wd read N-contiguous) and the dx GEMM
// ([dG|dU] x [Wg;Wu] with the weights read N-contiguous).
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_DGATED, false, true>(const Params&, int, cudaStream_t, bool);
template cudaError_t launch_gemm<EPI_DACT, false, true>(const Params&, int, cudaStream_t, bool);
template cudaError_t launch_gemm<EPI_STORE_BF16, false, true>(const Params&, int, cudaStream_t, bool);
}  // namespace mlpk
