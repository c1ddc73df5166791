// Decode-sized forward (one to four tokens) on the CUDA cores.  The
// library takes it for one or two tokens, where it streams the weights a
// few per cent faster than the warp-MMA stream (k_decode_mma.cu); from three
// tokens on its fused multiply-adds outrun the instruction issue.
//
// With a few tokens every weight element is used a few times: the forward
// is a weight stream, bound by HBM.  The tensor-core path reads its
// K-major weight boxes 128 bytes per row at a time, scattered over 128 rows,
// and streams at ~4 TB/s.  Here each warp owns whole weight rows and reads
// them front to back, 512 contiguous bytes per warp-wide 16-byte load, with
// the next group of loads issued before the current group is used
// (registers double-buffered), so every warp keeps its loads in flight
// continuously.  The token rows (x, or the postact for the down projection)
// are staged whole in shared memory once per CTA; each lane accumulates its
// share of the dot products in fp32, reduced across the warp at the end.
// Two CTAs per SM.
//
// One kernel, three epilogues (MODE):
//   DEC_GATED    y0 = x Wg^T, y1 = x Wu^T:  a = s*act(y0)*y1 (+ G = y0, U = y1)
//   DEC_NONGATED y0 = x W1^T:               a = s*act(y0)    (+ P = y0)
//   DEC_STORE    y0 = a Wd^T:               out = y0
// Rows are dealt to warps round-robin, block-minor (warp w of block b is
// warp number w * blocks + b, and takes rows number + j * warps), so that a
// last, partial round spreads over all blocks; each pass takes RPW rows of
// every weight matrix.
#include <atomic>

#include "act.cuh"
#include "gemm_params.h"
#include "ptx.cuh"

namespace mlpk {

enum DecMode : int { DEC_GATED = 0, DEC_NONGATED = 1, DEC_STORE = 2 };

constexpr int DEC_THREADS = 256;
constexpr int DEC_WARPS = DEC_THREADS / 32;
// CTAs per SM, rows of each weight matrix per warp and pass, and 16-byte
// chunks per lane in one load group (two groups in flight)
template <int MODE>
__host__ __device__ constexpr int dec_ctas() { return 2; }
// (the gated pass with three or four tokens takes one row per matrix, so
// that its weights, tokens and sums fit 128 registers)
template <int MODE, int MT>
__host__ __device__ constexpr int dec_rpw() { return MODE == DEC_GATED && MT > 2 ? 1 : 2; }
template <int MODE, int MT>
__host__ __device__ constexpr int dec_cpl() { return MODE == DEC_GATED && MT <= 2 ? 2 : 4; }

// 8 bf16 (one 16-byte vector) -> 8 floats (exact).
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}

// Streaming 16-byte load of weights that are read exactly once.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int MODE, int MT>
struct DecGroup {
  static constexpr int NMAT = MODE == DEC_GATED ? 2 : 1;
  static constexpr int RPW = dec_rpw<MODE, MT>();
  static constexpr int CPL = dec_cpl<MODE, MT>();
  uint4 w[CPL][NMAT][RPW];

  // the group's chunks: chunk (g * CPL + q) * 32 + lane of each row
  __device__ __forceinline__ void load(const __nv_bfloat16* const (&W)[2], const int (&row)[RPW],
                                       int R, int K, int g, int lane) {
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const int c = (g * CPL + q) * 32 + lane;
#pragma unroll
      for (int a = 0; a < NMAT; ++a)
#pragma unroll
        for (int j = 0; j < RPW; ++j)
          w[q][a][j] = (row[j] < R && 8 * c < K)
                           ? ld_stream_v4(W[a] + static_cast<size_t>(row[j]) * K + 8 * c)
                           : make_uint4(0, 0, 0, 0);
    }
  }

  // acc[a][j][m] += the group's part of row j of matrix a times token m
  // (chunks past the row end hold zeros and read token chunk 0)
  __device__ __forceinline__ void fma(const uint4* tok, int K, int g, int lane,
                                      float (&acc)[NMAT][RPW][MT]) const {
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      int c = (g * CPL + q) * 32 + lane;
      if (8 * c >= K) c = 0;
      float wf[NMAT][RPW][8];
#pragma unroll
      for (int a = 0; a < NMAT; ++a)
#pragma unroll
        for (int j = 0; j < RPW; ++j) bf16x8_to_f32(w[q][a][j], wf[a][j]);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float xf[8];
        bf16x8_to_f32(tok[m * (K / 8) + c], xf);
#pragma unroll
        for (int a = 0; a < NMAT; ++a)
#pragma unroll
          for (int j = 0; j < RPW; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[a][j][m] = fmaf(wf[a][j][e], xf[e], acc[a][j][m]);
      }
    }
  }
};

// The warp's rows of pass `pass`.
template <int RPW>
__device__ __forceinline__ void dec_rows(int gw, int nw, int pass, int (&row)[RPW]) {
#pragma unroll
  for (int j = 0; j < RPW; ++j) row[j] = gw + (pass * RPW + j) * nw;
}

template <int ACT, int MODE, int MT>
__global__ void __launch_bounds__(DEC_THREADS, dec_ctas<MODE>()) k_decode(
    const __nv_bfloat16* __restrict__ T, const __nv_bfloat16* __restrict__ W0,
    const __nv_bfloat16* __restrict__ W1, __nv_bfloat16* __restrict__ out,
    __nv_bfloat16* __restrict__ o1, __nv_bfloat16* __restrict__ o2, int M, int R, int K, float s,
    int passes, int* status) {
  using G = DecGroup<MODE, MT>;
  constexpr int NMAT = G::NMAT;
  // the call's status word (the first kernel of the call clears it)
  if (status != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *status = 0;
  constexpr int RPW = G::RPW;
  extern __shared__ uint4 tok[];  // [MT][K / 8], token rows m >= M as zeros
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = gridDim.x * DEC_WARPS;
  const int gw = warp * gridDim.x + blockIdx.x;
  const __nv_bfloat16* const W[2] = {W0, W1};
  const int ngroups = (K / 8 + 32 * G::CPL - 1) / (32 * G::CPL);
  // The warp's work is one sequence of load groups over all its passes
  // (step i = group i % ngroups of pass i / ngroups), with two groups in
  // flight throughout: the first groups of a pass are requested before the
  // previous pass's sums are reduced and stored.
  int npass = 0;
  if (gw < R) npass = min(passes, (R - gw + RPW * nw - 1) / (RPW * nw));
  const int nsteps = npass * ngroups;
  int rows_a[RPW], rows_b[RPW];  // rows of the steps in buffers A and B
  G ga, gb;
  // The weights do not depend on the previous kernel: the first two groups
  // are requested before waiting for it.
  if (nsteps > 0) {
    dec_rows<RPW>(gw, nw, 0, rows_a);
    ga.load(W, rows_a, R, K, 0, lane);
  }
  if (nsteps > 1) {
    dec_rows<RPW>(gw, nw, 1 / ngroups, rows_b);
    gb.load(W, rows_b, R, K, 1 % ngroups, lane);
  }
  // the tokens may be the previous kernel's output (the postact)
  pdl_wait();
  for (int idx = threadIdx.x; idx < MT * (K / 8); idx += DEC_THREADS) {
    const int m = idx / (K / 8), c = idx - m * (K / 8);
    tok[idx] = m < M ? ld_global_v4(T + static_cast<size_t>(m) * K + 8 * c) : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  pdl_launch_dependents();

  float acc[NMAT][RPW][MT];
  auto clear = [&] {
#pragma unroll
    for (int a = 0; a < NMAT; ++a)
#pragma unroll
      for (int j = 0; j < RPW; ++j)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[a][j][m] = 0.f;
  };
  // warp sums of a finished pass; lane j * MT + m stores (row j, token m)
  auto finish = [&](const int (&row)[RPW]) {
#pragma unroll
    for (int a = 0; a < NMAT; ++a)
#pragma unroll
      for (int j = 0; j < RPW; ++j)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          float v = acc[a][j][m];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          acc[a][j][m] = v;
        }
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (lane != j * MT + m || m >= M || row[j] >= R) continue;
        const size_t o = static_cast<size_t>(m) * R + row[j];
        const float y0 = acc[0][j][m];
        if constexpr (MODE == DEC_STORE) {
          out[o] = __float2bfloat16_rn(y0);
        } else if constexpr (MODE == DEC_GATED) {
          const float y1 = acc[NMAT - 1][j][m];
          out[o] = __float2bfloat16_rn(s * act_f<ACT>(y0) * y1);
          if (o1) o1[o] = __float2bfloat16_rn(y0);
          if (o2) o2[o] = __float2bfloat16_rn(y1);
        } else {
          out[o] = __float2bfloat16_rn(s * act_f<ACT>(y0));
          if (o1) o1[o] = __float2bfloat16_rn(y0);
        }
      }
    }
    clear();
  };

  clear();
  for (int i = 0; i < nsteps; i += 2) {
    // step i from buffer A (step i + 1 is in flight in buffer B)
    ga.fma(tok, K, i % ngroups, lane, acc);
    if (i % ngroups == ngroups - 1) finish(rows_a);
    if (i + 2 < nsteps) {
      dec_rows<RPW>(gw, nw, (i + 2) / ngroups, rows_a);
      ga.load(W, rows_a, R, K, (i + 2) % ngroups, lane);
    }
    if (i + 1 < nsteps) {
      // step i + 1 from buffer B (step i + 2 is in flight in buffer A)
      gb.fma(tok, K, (i + 1) % ngroups, lane, acc);
      if ((i + 1) % ngroups == ngroups - 1) finish(rows_b);
      if (i + 3 < nsteps) {
        dec_rows<RPW>(gw, nw, (i + 3) / ngroups, rows_b);
        gb.load(W, rows_b, R, K, (i + 3) % ngroups, lane);
      }
    }
  }
}

template <int ACT, int MODE, int MT>
cudaError_t launch_decode_inst(const __nv_bfloat16* T, const __nv_bfloat16* W0,
                               const __nv_bfloat16* W1, __nv_bfloat16* out, __nv_bfloat16* o1,
                               __nv_bfloat16* o2, int M, int R, int K, float s,
                               cudaStream_t stream, bool pdl, int* status) {
  auto kern = k_decode<ACT, MODE, MT>;
  constexpr int RPW = dec_rpw<MODE, MT>();
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // dec_ctas CTAs per SM, or fewer when the rows run out
  const int warps_needed = (R + RPW - 1) / RPW;
  int blocks = (warps_needed + DEC_WARPS - 1) / DEC_WARPS;
  if (blocks > dec_ctas<MODE>() * sms) blocks = dec_ctas<MODE>() * sms;
  if (blocks < 1) blocks = 1;
  const int nw = blocks * DEC_WARPS;
  const int passes = (R + nw * RPW - 1) / (nw * RPW);
  static std::atomic<unsigned> configured{0};  // devices that got the attribute
  if (dev >= 31 || !(configured.load() & (1u << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DECODE_MAX_TOKEN_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 31) configured.fetch_or(1u << dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(DEC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = MT * K * 2;  // the staged token rows
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, T, W0, W1, out, o1, o2, M, R, K, s, passes, status);
}

template <int ACT, int MODE>
cudaError_t launch_decode_mt(const void* T, const void* W0, const void* W1, void* out, void* o1,
                             void* o2, int M, int R, int K, float s, cudaStream_t stream,
                             bool pdl, int* status) {
  auto t = static_cast<const __nv_bfloat16*>(T);
  auto w0 = static_cast<const __nv_bfloat16*>(W0);
  auto w1 = static_cast<const __nv_bfloat16*>(W1);
  auto y = static_cast<__nv_bfloat16*>(out);
  auto y1 = static_cast<__nv_bfloat16*>(o1);
  auto y2 = static_cast<__nv_bfloat16*>(o2);
  switch (M) {
    case 1: return launch_decode_inst<ACT, MODE, 1>(t, w0, w1, y, y1, y2, M, R, K, s, stream, pdl, status);
    case 2: return launch_decode_inst<ACT, MODE, 2>(t, w0, w1, y, y1, y2, M, R, K, s, stream, pdl, status);
    case 3: return launch_decode_inst<ACT, MODE, 3>(t, w0, w1, y, y1, y2, M, R, K, s, stream, pdl, status);
    default: return launch_decode_inst<ACT, MODE, 4>(t, w0, w1, y, y1, y2, M, R, K, s, stream, pdl, status);
  }
}

cudaError_t launch_decode_act(const void* x, const void* Wg, const void* Wu, void* a, void* G,
                              void* U, int M, int H, int I, int act, bool gated, float s,
                              cudaStream_t stream, bool pdl, int* status) {
  if (gated) {
    switch (act) {
      case ACT_RELU: return launch_decode_mt<ACT_RELU, DEC_GATED>(x, Wg, Wu, a, G, U, M, I, H, s, stream, pdl, status);
      case ACT_GELU_TANH: return launch_decode_mt<ACT_GELU_TANH, DEC_GATED>(x, Wg, Wu, a, G, U, M, I, H, s, stream, pdl, status);
      case ACT_SIGMOID: return launch_decode_mt<ACT_SIGMOID, DEC_GATED>(x, Wg, Wu, a, G, U, M, I, H, s, stream, pdl, status);
      default: return launch_decode_mt<ACT_SILU, DEC_GATED>(x, Wg, Wu, a, G, U, M, I, H, s, stream, pdl, status);
    }
  }
  switch (act) {
    case ACT_RELU: return launch_decode_mt<ACT_RELU, DEC_NONGATED>(x, Wg, nullptr, a, G, nullptr, M, I, H, s, stream, pdl, status);
    case ACT_GELU_TANH: return launch_decode_mt<ACT_GELU_TANH, DEC_NONGATED>(x, Wg, nullptr, a, G, nullptr, M, I, H, s, stream, pdl, status);
    default: return launch_decode_mt<ACT_RELU_SQ, DEC_NONGATED>(x, Wg, nullptr, a, G, nullptr, M, I, H, s, stream, pdl, status);
  }
}

cudaError_t launch_decode_down(const void* a, const void* Wd, void* out, int M, int H, int I,
                               cudaStream_t stream, bool pdl) {
  return launch_decode_mt<0, DEC_STORE>(a, Wd, nullptr, out, nullptr, nullptr, M, H, I, 1.f,
                                        stream, pdl, nullptr);
}

}  // namespace mlpk
