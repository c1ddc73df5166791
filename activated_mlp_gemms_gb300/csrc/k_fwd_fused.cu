// The gated forward in one launch (EPI_FWD_FUSED): the gate/up tiles with
// the gated activation epilogue, then the down projection tiles of each
// 256-row block once its postact is stored.  CTA pairs only.
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_FWD_FUSED, false, false, 2, ACT_SILU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_FWD_FUSED, false, false, 2, ACT_SILU>();
template cudaError_t launch_gemm<EPI_FWD_FUSED, false, false, 2, ACT_RELU>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_FWD_FUSED, false, false, 2, ACT_RELU>();
template cudaError_t launch_gemm<EPI_FWD_FUSED, false, false, 2, ACT_GELU_TANH>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_FWD_FUSED, false, false, 2, ACT_GELU_TANH>();
template cudaError_t launch_gemm<EPI_FWD_FUSED, false, false, 2, ACT_SIGMOID>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_FWD_FUSED, false, false, 2, ACT_SIGMOID>();
}  // namespace mlpk
