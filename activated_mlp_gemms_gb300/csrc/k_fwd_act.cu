// Forward fc1 kernel instances with the non-gated activation epilogue
// (relu^2, tanh-GELU, relu); operands K-major.
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_ACT_FWD, false, false, 1, ACT_RELU_SQ>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACT_FWD, false, false, 1, ACT_RELU_SQ>();
template cudaError_t launch_gemm<EPI_ACT_FWD, false, false, 2, ACT_RELU_SQ>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACT_FWD, false, false, 2, ACT_RELU_SQ>();
template cudaError_t launch_gemm<EPI_ACT_FWD, false, false, 1, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACT_FWD, false, false, 1, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_ACT_FWD, false, false, 2, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACT_FWD, false, false, 2, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_ACT_FWD, false, false, 1, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACT_FWD, false, false, 1, ACT_RELU>();
template cudaError_t launch_gemm<EPI_ACT_FWD, false, false, 2, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACT_FWD, false, false, 2, ACT_RELU>();
}  // namespace mlpk
