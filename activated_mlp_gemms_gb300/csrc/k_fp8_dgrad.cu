// Backward GEMMs of the 8-bit ReLU^2 MLP with a K-major A and an MN-major B:
// the e5m2 derivative (dout8 times the W2 codes read MN-major, ReLU^2' from
// the saved bf16 preact, re-quantised to e5m2 with its amax) and dx (the
// derivative codes times the W1 codes read MN-major, dequantised to bf16).
#include "gemm.cuh"

namespace mlpk {

template cudaError_t launch_gemm<EPI_DGRAD_F8, false, true, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGRAD_F8, false, true, 1, 0>();
template cudaError_t launch_gemm<EPI_DGRAD_F8, false, true, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGRAD_F8, false, true, 2, 0>();
template cudaError_t launch_gemm<EPI_STORE_BF16_F8, false, true, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16_F8, false, true, 1, 0>();
template cudaError_t launch_gemm<EPI_STORE_BF16_F8, false, true, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16_F8, false, true, 2, 0>();

}  // namespace mlpk
