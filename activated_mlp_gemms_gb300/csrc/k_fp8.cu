// 8-bit (FP8) kernels of the ReLU^2 MLP forward: the quantisation of bf16
// tensors to e4m3 or e5m2 codes with a dequant scale (and their amax), and
// the forward GEMM instances: fc1 with the ReLU^2 epilogue that re-quantises
// its output, and the down projection with a dequantising bf16 store.
#include "gemm.cuh"

namespace mlpk {

// q = f8(fp32(x * fp32(1 / *scale))), saturating, 8 values (one 16-byte
// load, one 8-byte store) per vector; each thread loads four grid-strided
// vectors before converting them, so that their loads are in flight
// together.  |x|'s maximum goes to *amax.
template <int FMT>
__device__ __forceinline__ uint2 quant8(uint4 v, float inv, float& mx) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[2] = {0, 0};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = unpack_bf16x2(w[j]);
    mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
    const uint16_t c = FMT == F8_E5M2 ? pack_e5m2x2(f.x * inv, f.y * inv)
                                      : pack_e4m3x2(f.x * inv, f.y * inv);
    o[j >> 1] |= static_cast<uint32_t>(c) << (16 * (j & 1));
  }
  return make_uint2(o[0], o[1]);
}

template <int FMT>
__global__ void __launch_bounds__(256) k_quant_f8(const __nv_bfloat16* __restrict__ src,
                                                  long long n8, const float* __restrict__ scale,
                                                  uint8_t* __restrict__ dst, float* amax) {
  pdl_wait();
  pdl_launch_dependents();
  const float inv = 1.0f / *scale;
  float mx = 0.f;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = (i + u * stride < n8) ? ld_global_v4(src + 8 * (i + u * stride)) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * stride < n8)
        *reinterpret_cast<uint2*>(dst + 8 * (i + u * stride)) = quant8<FMT>(v[u], inv, mx);
  }
  if (amax) {
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    if ((threadIdx.x & 31) == 0 && mx > 0.f) atomicMax(reinterpret_cast<int*>(amax), __float_as_int(mx));
  }
}

cudaError_t launch_quant_f8(const void* src, long long n, const float* scale, void* dst,
                            float* amax, int fmt, cudaStream_t stream, bool pdl) {
  const long long n8 = n / 8;  // n is a multiple of 8
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (n8 + 255) / 256;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  auto s = static_cast<const __nv_bfloat16*>(src);
  auto d = static_cast<uint8_t*>(dst);
  if (fmt == F8_E5M2) return cudaLaunchKernelEx(&cfg, k_quant_f8<F8_E5M2>, s, n8, scale, d, amax);
  return cudaLaunchKernelEx(&cfg, k_quant_f8<F8_E4M3>, s, n8, scale, d, amax);
}

// The delayed-scale refresh of gpt.py (_refresh_delayed_scale): per slot i,
// a = max of the slot's `width` amax values (a NaN among them makes the
// max NaN, as torch's amax does), NaN and +-inf read as 0 (nan_to_num), a
// clamped to at most 1e12; the scale becomes max(a * gain, floor) when
// a > 0 and keeps its value otherwise; the amax values are cleared.  One
// thread per slot.
__global__ void __launch_bounds__(128) k_refresh_scales(float* amax, float* scale, int n,
                                                        int width, float gain, float floor_v) {
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float* row = amax + static_cast<long long>(i) * width;
  float a = row[0];
  for (int j = 1; j < width; ++j) {
    const float v = row[j];
    a = (isnan(a) || isnan(v)) ? __int_as_float(0x7fc00000) : fmaxf(a, v);
  }
  if (!isfinite(a)) a = 0.f;
  a = fminf(a, 1e12f);
  if (a > 0.f) scale[i] = fmaxf(a * gain, floor_v);
  for (int j = 0; j < width; ++j) row[j] = 0.f;
}

cudaError_t launch_refresh_scales(float* amax, float* scale, int n, int width, float gain,
                                  float floor_v, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n + 127) / 128), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_refresh_scales, amax, scale, n, width, gain, floor_v);
}

template cudaError_t launch_gemm<EPI_ACT_FWD_F8, false, false, 1, ACT_RELU_SQ>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACT_FWD_F8, false, false, 1, ACT_RELU_SQ>();
template cudaError_t launch_gemm<EPI_ACT_FWD_F8, false, false, 2, ACT_RELU_SQ>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_ACT_FWD_F8, false, false, 2, ACT_RELU_SQ>();
template cudaError_t launch_gemm<EPI_STORE_BF16_F8, false, false, 1, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16_F8, false, false, 1, 0>();
template cudaError_t launch_gemm<EPI_STORE_BF16_F8, false, false, 2, 0>(const Params&, int, cudaStream_t, bool);
template int max_groups<EPI_STORE_BF16_F8, false, false, 2, 0>();

}  // namespace mlpk
