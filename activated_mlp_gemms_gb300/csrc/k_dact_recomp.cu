// Fused recompute + derivative kernel instances (non-gated backward without
// saved preacts): x W1^T and dout Wd in one tile, epilogue a and dP, one per
// non-gated activation.
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_DACT_RECOMP, false, false, 1, ACT_RELU_SQ>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT_RECOMP, false, false, 1, ACT_RELU_SQ>();
template cudaError_t launch_gemm<EPI_DACT_RECOMP, false, false, 2, ACT_RELU_SQ>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT_RECOMP, false, false, 2, ACT_RELU_SQ>();
template cudaError_t launch_gemm<EPI_DACT_RECOMP, false, false, 1, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT_RECOMP, false, false, 1, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_DACT_RECOMP, false, false, 2, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT_RECOMP, false, false, 2, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_DACT_RECOMP, false, false, 1, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT_RECOMP, false, false, 1, ACT_RELU>();
template cudaError_t launch_gemm<EPI_DACT_RECOMP, false, false, 2, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DACT_RECOMP, false, false, 2, ACT_RELU>();
}  // namespace mlpk
