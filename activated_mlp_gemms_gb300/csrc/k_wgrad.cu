// Weight-gradient kernel instances: both operands MN-major (dW = D^T X with
// D [M,N'] and X [M,K'] row-major, reduced over the token dimension M).
// bf16 store, or fp32 in-place accumulation (atomic adds, split-K safe).
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_STORE_BF16, true, true, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16, true, true, 1, 0>();
template cudaError_t launch_gemm<EPI_STORE_BF16, true, true, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16, true, true, 2, 0>();
template cudaError_t launch_gemm<EPI_ACCUM_F32, true, true, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACCUM_F32, true, true, 1, 0>();
template cudaError_t launch_gemm<EPI_ACCUM_F32, true, true, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACCUM_F32, true, true, 2, 0>();
}  // namespace mlpk
