// The 8-bit derivative GEMM with the preact recomputed in the same tile:
// x8 W1_8^T (K-major B) and dout8 W2_8 (MN-major B) in the two accumulators,
// the e5m2 derivative codes and their amax from the epilogue.
#include "gemm.cuh"

namespace mlpk {

template cudaError_t launch_gemm<EPI_DGRAD_F8_RECOMP, false, false, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGRAD_F8_RECOMP, false, false, 1, 0>();
template cudaError_t launch_gemm<EPI_DGRAD_F8_RECOMP, false, false, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_DGRAD_F8_RECOMP, false, false, 2, 0>();

}  // namespace mlpk
