// Per-token kernels of the MLP block's neighbours (modded-nanogpt gpt.py,
// "process mlp": mlp_in = norm(x), then the scaled residual add):
//   k_rstd         rstd[m] = 1 / sqrt(mean_h x[m,h]^2 + eps)  (the RMS norm's
//                  scale, applied to the gate/up accumulators in their epilogue)
//   k_rmsnorm_bwd  dx = alpha dy + D - (rstd^2 / H) (sum_h D x) x, per token,
//                  in place over D (the dx GEMM's output, dn * rstd): the RMS
//                  norm's derivative plus the residual branch's gradient.
// One warp per token: each lane walks the row 8 bf16 (16 bytes) at a time,
// four steps unrolled so that their loads are in flight together; the row
// sums meet through warp shuffles in fp32.  HBM-bound.
#include "gemm_params.h"
#include "ptx.cuh"

namespace mlpk {

constexpr int ROW_WARPS = 8;  // tokens per 256-thread block

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(32 * ROW_WARPS) k_rstd(const __nv_bfloat16* __restrict__ x,
                                                         float* __restrict__ rstd, int M, int H,
                                                         float eps) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x * ROW_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;  // warp-uniform
  const __nv_bfloat16* xr = x + static_cast<size_t>(row) * H;
  float ss = 0.f;
#pragma unroll 4
  for (int c = 8 * lane; c < H; c += 256) {
    const uint4 v = ld_global_v4(xr + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      ss += f.x * f.x + f.y * f.y;
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) rstd[row] = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
}

__global__ void __launch_bounds__(32 * ROW_WARPS) k_rmsnorm_bwd(
    __nv_bfloat16* __restrict__ dx, const __nv_bfloat16* __restrict__ x,
    const __nv_bfloat16* __restrict__ dy, const float* __restrict__ rstd, int M, int H,
    float alpha) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x * ROW_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const size_t off = static_cast<size_t>(row) * H;
  float t = 0.f;  // sum_h D x
#pragma unroll 4
  for (int c = 8 * lane; c < H; c += 256) {
    const uint4 dv = ld_global_v4(dx + off + c), xv = ld_global_v4(x + off + c);
    const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w}, xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 d = unpack_bf16x2(dw[j]), xx = unpack_bf16x2(xw[j]);
      t += d.x * xx.x + d.y * xx.y;
    }
  }
  t = warp_sum(t);
  const float r = rstd[row];
  const float k = r * r * t / static_cast<float>(H);
#pragma unroll 4
  for (int c = 8 * lane; c < H; c += 256) {
    const uint4 dv = ld_global_v4(dx + off + c), xv = ld_global_v4(x + off + c),
                yv = ld_global_v4(dy + off + c);
    const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w}, xw[4] = {xv.x, xv.y, xv.z, xv.w},
                   yw[4] = {yv.x, yv.y, yv.z, yv.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 d = unpack_bf16x2(dw[j]), xx = unpack_bf16x2(xw[j]), g = unpack_bf16x2(yw[j]);
      o[j] = pack_bf16x2(alpha * g.x + d.x - k * xx.x, alpha * g.y + d.y - k * xx.y);
    }
    st_global_v4(dx + off + c, make_uint4(o[0], o[1], o[2], o[3]));
  }
}

namespace {
cudaLaunchConfig_t row_cfg(int M, cudaStream_t stream, bool pdl, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((M + ROW_WARPS - 1) / ROW_WARPS), 1, 1);
  cfg.blockDim = dim3(32 * ROW_WARPS, 1, 1);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}
}  // namespace

cudaError_t launch_rstd(const void* x, float* rstd, int M, int H, float eps, cudaStream_t stream,
                        bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = row_cfg(M, stream, pdl, attr);
  return cudaLaunchKernelEx(&cfg, k_rstd, static_cast<const __nv_bfloat16*>(x), rstd, M, H, eps);
}

cudaError_t launch_rmsnorm_bwd(void* dx, const void* x, const void* dy, const float* rstd, int M,
                               int H, float alpha, cudaStream_t stream, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = row_cfg(M, stream, pdl, attr);
  return cudaLaunchKernelEx(&cfg, k_rmsnorm_bwd, static_cast<__nv_bfloat16*>(dx),
                            static_cast<const __nv_bfloat16*>(x),
                            static_cast<const __nv_bfloat16*>(dy), rstd, M, H, alpha);
}

}  // namespace mlpk
