// Forward-pass kernel instances: fused gate/up (SwiGLU), fused non-gated
// fc1 + activation, and the plain bf16 GEMM of the down projection.
// Operands are K-major.
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_GATED_FWD, false, false>(const Params&, int, cudaStream_t, bool);
template cudaError_t launch_gemm<EPI_ACT_FWD, false, false>(const Params&, int, cudaStream_t, bool);
template cudaError_t launch_gemm<EPI_STORE_BF16, false, false>(const Params&, int, cudaStream_t, bool);
}  // namespace mlpk
