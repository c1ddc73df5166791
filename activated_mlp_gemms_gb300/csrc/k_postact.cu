// Elementwise postact a = s * act(G) * U (U == nullptr: s * act(G)), used when
// the backward pass needs only dWd: the postact is rebuilt from the saved or
// recomputed preacts without the activation derivative.  HBM-bound: 8 bf16
// per thread per step (16-byte loads and stores), grid-stride loop.
#include "act.cuh"
#include "ptx.cuh"

namespace mlpk {

template <int ACT, bool GATED>
__global__ void __launch_bounds__(256) k_postact(const __nv_bfloat16* __restrict__ G,
                                                 const __nv_bfloat16* __restrict__ U,
                                                 __nv_bfloat16* __restrict__ a, long long n8,
                                                 float s) {
  pdl_wait();
  pdl_launch_dependents();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8;
       i += (long long)gridDim.x * blockDim.x) {
    uint4 gv = ld_global_v4(G + 8 * i);
    uint4 uv = GATED ? ld_global_v4(U + 8 * i) : make_uint4(0, 0, 0, 0);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 g = unpack_bf16x2(gw[j]);
      float a0 = s * act_f<ACT>(g.x), a1 = s * act_f<ACT>(g.y);
      if (GATED) {
        float2 u = unpack_bf16x2(uw[j]);
        a0 *= u.x;
        a1 *= u.y;
      }
      o[j] = pack_bf16x2(a0, a1);
    }
    st_global_v4(a + 8 * i, make_uint4(o[0], o[1], o[2], o[3]));
  }
}

cudaError_t launch_postact(const void* G, const void* U, void* a, long long n, int act,
                           float scale, cudaStream_t stream, bool pdl) {
  const long long n8 = n / 8;  // n is a multiple of 8 (I % 8 == 0)
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
  auto g = static_cast<const __nv_bfloat16*>(G);
  auto u = static_cast<const __nv_bfloat16*>(U);
  auto o = static_cast<__nv_bfloat16*>(a);
  // `act` is the device activation (see Act); `gated` selects the times-U form
  if (U) {
    if (act == ACT_RELU) return cudaLaunchKernelEx(&cfg, k_postact<ACT_RELU, true>, g, u, o, n8, scale);
    if (act == ACT_GELU_TANH)
      return cudaLaunchKernelEx(&cfg, k_postact<ACT_GELU_TANH, true>, g, u, o, n8, scale);
    if (act == ACT_SIGMOID)
      return cudaLaunchKernelEx(&cfg, k_postact<ACT_SIGMOID, true>, g, u, o, n8, scale);
    return cudaLaunchKernelEx(&cfg, k_postact<ACT_SILU, true>, g, u, o, n8, scale);
  }
  if (act == ACT_RELU) return cudaLaunchKernelEx(&cfg, k_postact<ACT_RELU, false>, g, u, o, n8, scale);
  if (act == ACT_GELU_TANH)
    return cudaLaunchKernelEx(&cfg, k_postact<ACT_GELU_TANH, false>, g, u, o, n8, scale);
  return cudaLaunchKernelEx(&cfg, k_postact<ACT_RELU_SQ, false>, g, u, o, n8, scale);
}

// fp32 -> bf16 over n elements, 8 per thread per step (two 16-byte loads,
// one 16-byte store); the split-K partial sums of a decode-sized output,
// plus alpha * resid when a residual is given.
__global__ void __launch_bounds__(256) k_f32_to_bf16(const float* __restrict__ src,
                                                     __nv_bfloat16* __restrict__ dst, long long n8,
                                                     const __nv_bfloat16* __restrict__ resid,
                                                     float alpha) {
  pdl_wait();
  pdl_launch_dependents();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 a = ld_global_v4(src + 8 * i);
    const uint4 b = ld_global_v4(src + 8 * i + 4);
    float v[8] = {__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z),
                  __uint_as_float(a.w), __uint_as_float(b.x), __uint_as_float(b.y),
                  __uint_as_float(b.z), __uint_as_float(b.w)};
    if (resid) {
      const uint4 r = ld_global_v4(resid + 8 * i);
      const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = unpack_bf16x2(rw[j]);
        v[2 * j] += alpha * f.x;
        v[2 * j + 1] += alpha * f.y;
      }
    }
    st_global_v4(dst + 8 * i, make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                         pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7])));
  }
}

cudaError_t launch_f32_to_bf16(const float* src, void* dst, long long n, cudaStream_t stream,
                               bool pdl, const void* resid, float alpha) {
  const long long n8 = n / 8;
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
  return cudaLaunchKernelEx(&cfg, k_f32_to_bf16, src, static_cast<__nv_bfloat16*>(dst), n8,
                            static_cast<const __nv_bfloat16*>(resid), alpha);
}

}  // namespace mlpk
