// Weight gradients of the 8-bit ReLU^2 MLP: both operands MN-major (the
// token dimension is the reduction), dequantised to bf16; one grouped launch
// computes dW1 and dW2.
#include "gemm.cuh"

namespace mlpk {

template cudaError_t launch_gemm<EPI_STORE_BF16_F8, true, true, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16_F8, true, true, 1, 0>();
template cudaError_t launch_gemm<EPI_STORE_BF16_F8, true, true, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16_F8, true, true, 2, 0>();

}  // namespace mlpk
