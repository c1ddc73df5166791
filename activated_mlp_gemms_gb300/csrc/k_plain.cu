// Plain GEMM instances: the down projection (both operands K-major) and dx
// ([dG|dU] x [Wg;Wu], B read N-contiguous), with the bf16 store epilogue and,
// for decode-sized token counts, the fp32 split-K accumulate epilogue.
#include "gemm.cuh"

namespace mlpk {
template cudaError_t launch_gemm<EPI_STORE_BF16, false, false, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16, false, false, 1, 0>();
template cudaError_t launch_gemm<EPI_STORE_BF16, false, false, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16, false, false, 2, 0>();
template cudaError_t launch_gemm<EPI_STORE_BF16, false, true, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16, false, true, 1, 0>();
template cudaError_t launch_gemm<EPI_STORE_BF16, false, true, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16, false, true, 2, 0>();
template cudaError_t launch_gemm<EPI_ACCUM_F32, false, false, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACCUM_F32, false, false, 1, 0>();
template cudaError_t launch_gemm<EPI_ACCUM_F32, false, false, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACCUM_F32, false, false, 2, 0>();
template cudaError_t launch_gemm<EPI_ACCUM_F32, false, true, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACCUM_F32, false, true, 1, 0>();
template cudaError_t launch_gemm<EPI_ACCUM_F32, false, true, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACCUM_F32, false, true, 2, 0>();
}  // namespace mlpk
