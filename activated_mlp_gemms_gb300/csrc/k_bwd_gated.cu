// dgated kernel instances (dout x Wd with Wd read N-contiguous, epilogue
// dG, dU and the postact), one per gate activation.
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_DGATED, false, true, 1, ACT_SILU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGATED, false, true, 1, ACT_SILU>();
template cudaError_t launch_gemm<EPI_DGATED, false, true, 2, ACT_SILU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGATED, false, true, 2, ACT_SILU>();
template cudaError_t launch_gemm<EPI_DGATED, false, true, 1, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGATED, false, true, 1, ACT_RELU>();
template cudaError_t launch_gemm<EPI_DGATED, false, true, 2, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGATED, false, true, 2, ACT_RELU>();
template cudaError_t launch_gemm<EPI_DGATED, false, true, 1, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGATED, false, true, 1, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_DGATED, false, true, 2, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGATED, false, true, 2, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_DGATED, false, true, 1, ACT_SIGMOID>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGATED, false, true, 1, ACT_SIGMOID>();
template cudaError_t launch_gemm<EPI_DGATED, false, true, 2, ACT_SIGMOID>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGATED, false, true, 2, ACT_SIGMOID>();
}  // namespace mlpk
