// dact kernel instances (dout x Wd with Wd read N-contiguous, epilogue dP
// and the postact), one per non-gated activation.
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_DACT, false, true, 1, ACT_RELU_SQ>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT, false, true, 1, ACT_RELU_SQ>();
template cudaError_t launch_gemm<EPI_DACT, false, true, 2, ACT_RELU_SQ>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT, false, true, 2, ACT_RELU_SQ>();
template cudaError_t launch_gemm<EPI_DACT, false, true, 1, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT, false, true, 1, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_DACT, false, true, 2, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT, false, true, 2, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_DACT, false, true, 1, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT, false, true, 1, ACT_RELU>();
template cudaError_t launch_gemm<EPI_DACT, false, true, 2, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT, false, true, 2, ACT_RELU>();
}  // namespace mlpk
