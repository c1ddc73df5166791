// Forward gate/up kernel instances with the gated activation epilogue
// (silu, relu, tanh-GELU or sigmoid on the gate, times the up projection);
// operands K-major.
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false, 1, ACT_SILU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_GATED_FWD, false, false, 1, ACT_SILU>();
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false, 2, ACT_SILU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_GATED_FWD, false, false, 2, ACT_SILU>();
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false, 1, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_GATED_FWD, false, false, 1, ACT_RELU>();
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false, 2, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_GATED_FWD, false, false, 2, ACT_RELU>();
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false, 1, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_GATED_FWD, false, false, 1, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false, 2, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_GATED_FWD, false, false, 2, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false, 1, ACT_SIGMOID>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_GATED_FWD, false, false, 1, ACT_SIGMOID>();
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false, 2, ACT_SIGMOID>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_GATED_FWD, false, false, 2, ACT_SIGMOID>();
}  // namespace mlpk
