// Forward-pass kernel instances: fused gate/up (SwiGLU), fused non-gated
// fc1 + activation, and the plain bf16 GEMM of the down projection.
// Operands are K-major.
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false, 1>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_GATED_FWD, false, false, 1>();
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false, 2>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_GATED_FWD, false, false, 2>();
template cudaError_t launch_gemm<EPI_ACT_FWD, false, false, 1>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACT_FWD, false, false, 1>();
template cudaError_t launch_gemm<EPI_ACT_FWD, false, false, 2>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACT_FWD, false, false, 2>();
template cudaError_t launch_gemm<EPI_STORE_BF16, false, false, 1>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16, false, false, 1>();
template cudaError_t launch_gemm<EPI_STORE_BF16, false, false, 2>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16, false, false, 2>();
}  // namespace mlpk
