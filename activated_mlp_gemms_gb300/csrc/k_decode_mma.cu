// Decode-sized forward (up to sixteen tokens): a weight stream whose dot
// products run on the warp-level MMA (mma.sync m16n8k16, bf16 in, fp32
// accumulate).  The library takes it for three to eight tokens; with 9-16
// (two 8-token blocks, twice the token loads) it is no faster than the
// tensor-core GEMMs, and the 16-token instances run only when a test forces
// them.
//
// With M <= 16 tokens the forward reads every weight once and does M
// multiply-adds per weight element, so it is bound by HBM, not by any
// arithmetic unit.  On the CUDA cores every weight element costs a bf16 ->
// fp32 conversion and, per token, a token conversion and a fused
// multiply-add; at four tokens that already outruns the instruction issue.
// The warp-level MMA takes a 16-row x 16-k weight fragment and a 16-k x
// 8-token fragment straight from registers: one 16-byte weight load per lane
// feeds two MMAs, and the kernel issues about 12 instructions per 2 KB of
// weights.
//
// Fragments without shuffles.  The MMA's k index is a summation index, so
// any permutation of k that A and B share gives the same dot products.  Lane
// (g = lane / 4, q = lane % 4) loads 16 bytes (8 consecutive k) of weight
// rows g and g + 8 and of token g, all at k0 + 8q; elements 0-3 of the
// three loads form the fragments of one MMA, elements 4-7 those of the
// next.  Within one k-step of 32 the four lanes of a row read its 64 bytes
// contiguously; a load group of two k-steps reads 128 bytes of each of the
// 16 rows.
//
// Work.  A CTA owns 16 consecutive weight rows (of Wg and Wu for the gated
// pass; 32, two 16-row tiles per warp, for the down pass with 16 tokens, so
// that each token fragment feeds twice the weights: 36 -> 30 us for
// Llama-3-8B's Wd) and all of K; its S warps take the 64-wide k groups
// round-robin (warp w: groups w, w + S, ...), with two groups in flight per
// warp (registers double-buffered).  S is the most warps with which the
// whole grid is resident at once (md_warps).  The warps' partial sums meet
// in shared memory; the CTA's first warp applies the epilogue.  The token rows are
// read through L1/L2 (they are small and every CTA reads them); the weights
// with no L1 allocation (each is read once).  The weights do not depend on
// the previous kernel, so the first group's weights are requested before
// waiting for it.
//
// Epilogues (MODE, as the CUDA-core decode kernel's):
//   MD_GATED    y0 = x Wg^T, y1 = x Wu^T:  a = s*act(y0)*y1 (+ G = y0, U = y1)
//   MD_NONGATED y0 = x W1^T:               a = s*act(y0)    (+ P = y0)
//   MD_STORE    y0 = a Wd^T:               out = y0
#include <atomic>

#include "act.cuh"
#include "gemm_params.h"
#include "ptx.cuh"

namespace mlpk {

namespace {

enum MmaDecMode : int { MD_GATED = 0, MD_NONGATED = 1, MD_STORE = 2 };

constexpr int MD_MAX_WARPS = 16;
// threads per CTA at most: 16 warps (128 registers a thread), the gated
// pass 8 (its two weight matrices need more than 128 with 16 tokens)
template <int MODE>
__host__ __device__ constexpr int md_max_threads() { return MODE == MD_GATED ? 256 : 512; }
constexpr int MD_ROWS = 16;  // weight rows of one MMA tile (the MMA's M)
// 16-row tiles per warp: two for the down pass with 16 tokens, so that each
// token fragment it loads feeds twice the weights
template <int MODE, int NT>
__host__ __device__ constexpr int md_row_tiles() { return (MODE == MD_STORE && NT == 16) ? 2 : 1; }
constexpr int MD_KG = 64;    // k per load group (two k-steps of 32)

__device__ __forceinline__ uint4 ld_weights_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_tokens_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// d += A (16 x 16, row-major fragment a0..a3) * B (16 x 8, column-major
// fragment b0, b1), bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int MODE, int NT, int RT>
struct MdGroup {
  static constexpr int NMAT = MODE == MD_GATED ? 2 : 1;
  static constexpr int NTB = NT / 8;  // 8-token blocks
  uint4 w[NMAT][RT][2][2];            // [matrix][16-row tile][row g, g + 8][k-step]
  uint4 t[NTB][2];                    // [token block][k-step]

  // the weights of the group starting at k0 (zeros past the rows or K)
  __device__ __forceinline__ void load_w(const __nv_bfloat16* const (&W)[2], int row0, int R,
                                         int K, int k0, int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int k = k0 + 32 * s + 8 * q;
#pragma unroll
      for (int a = 0; a < NMAT; ++a)
#pragma unroll
        for (int rt = 0; rt < RT; ++rt)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int r = row0 + 16 * rt + g + 8 * h;
            w[a][rt][h][s] = (k < K && r < R)
                                 ? ld_weights_v4(W[a] + static_cast<size_t>(r) * K + k)
                                 : make_uint4(0, 0, 0, 0);
          }
    }
  }

  // the token chunks of the group (zeros past the M tokens or K)
  __device__ __forceinline__ void load_t(const __nv_bfloat16* T, int M, int K, int k0, int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int k = k0 + 32 * s + 8 * q;
#pragma unroll
      for (int b = 0; b < NTB; ++b) {
        const int m = 8 * b + g;
        t[b][s] = (k < K && m < M) ? ld_tokens_v4(T + static_cast<size_t>(m) * K + k)
                                   : make_uint4(0, 0, 0, 0);
      }
    }
  }

  // acc[a][rt][b] += the group's part of rows (g, g + 8) of tile rt of
  // matrix a times tokens of block b
  __device__ __forceinline__ void mma(float (&acc)[NMAT][RT][NTB][4]) const {
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int a = 0; a < NMAT; ++a)
#pragma unroll
        for (int rt = 0; rt < RT; ++rt)
#pragma unroll
          for (int b = 0; b < NTB; ++b) {
            const uint4(&x)[2][2] = w[a][rt];
            mma_16816(acc[a][rt][b], x[0][s].x, x[1][s].x, x[0][s].y, x[1][s].y, t[b][s].x,
                      t[b][s].y);
            mma_16816(acc[a][rt][b], x[0][s].z, x[1][s].z, x[0][s].w, x[1][s].w, t[b][s].z,
                      t[b][s].w);
          }
  }
};

template <int ACT, int MODE, int NT>
__global__ void __launch_bounds__(md_max_threads<MODE>()) k_decode_mma(
    const __nv_bfloat16* __restrict__ T, const __nv_bfloat16* __restrict__ W0,
    const __nv_bfloat16* __restrict__ W1, __nv_bfloat16* __restrict__ out,
    __nv_bfloat16* __restrict__ o1, __nv_bfloat16* __restrict__ o2, int M, int R, int K, float s,
    int* status) {
  constexpr int RT = md_row_tiles<MODE, NT>();
  using G = MdGroup<MODE, NT, RT>;
  // the call's status word (the first kernel of the call clears it)
  if (status != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *status = 0;
  constexpr int NMAT = G::NMAT, NTB = G::NTB;
  constexpr int DEPTH = 2;  // load groups in flight per warp (deeper: no faster, more registers)
  // the warps' partial sums, [warp][matrix][token block][lane] x 4 floats
  __shared__ float4 part[md_max_threads<MODE>() / 32][NMAT][RT][NTB][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int row0 = blockIdx.x * MD_ROWS * RT;
  const __nv_bfloat16* const W[2] = {W0, W1};
  const int ngroups = (K + MD_KG - 1) / MD_KG;

  float acc[NMAT][RT][NTB][4];
#pragma unroll
  for (int a = 0; a < NMAT; ++a)
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int b = 0; b < NTB; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[a][rt][b][e] = 0.f;

  // groups warp, warp + nwarps, ... in a ring of DEPTH register buffers
  G buf[DEPTH];
  if (warp < ngroups) buf[0].load_w(W, row0, R, K, warp * MD_KG, lane);
  // the tokens may be the previous kernel's output (the postact)
  pdl_wait();
  if (warp < ngroups) buf[0].load_t(T, M, K, warp * MD_KG, lane);
#pragma unroll
  for (int j = 1; j < DEPTH; ++j) {
    const int gj = warp + j * nwarps;
    if (gj < ngroups) {
      buf[j].load_w(W, row0, R, K, gj * MD_KG, lane);
      buf[j].load_t(T, M, K, gj * MD_KG, lane);
    }
  }
  pdl_launch_dependents();
  for (int gi = warp; gi < ngroups;) {
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) {
      if (gi < ngroups) {
        buf[j].mma(acc);
        const int nx = gi + DEPTH * nwarps;
        if (nx < ngroups) {
          buf[j].load_w(W, row0, R, K, nx * MD_KG, lane);
          buf[j].load_t(T, M, K, nx * MD_KG, lane);
        }
      }
      gi += nwarps;
    }
  }

#pragma unroll
  for (int a = 0; a < NMAT; ++a)
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int b = 0; b < NTB; ++b)
        part[warp][a][rt][b][lane] = make_float4(acc[a][rt][b][0], acc[a][rt][b][1],
                                                 acc[a][rt][b][2], acc[a][rt][b][3]);
  __syncthreads();
  if (warp != 0) return;
  // the CTA's sums, in the accumulator layout: element (h, e) of lane
  // (g, q) is row 16 rt + g + 8h, token 2q + e of the block
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
    float y[NMAT][NTB][4];
#pragma unroll
    for (int a = 0; a < NMAT; ++a)
#pragma unroll
      for (int b = 0; b < NTB; ++b) {
        float4 v = part[0][a][rt][b][lane];
        for (int w2 = 1; w2 < nwarps; ++w2) {
          const float4 u = part[w2][a][rt][b][lane];
          v.x += u.x;
          v.y += u.y;
          v.z += u.z;
          v.w += u.w;
        }
        y[a][b][0] = v.x;
        y[a][b][1] = v.y;
        y[a][b][2] = v.z;
        y[a][b][3] = v.w;
      }
#pragma unroll
    for (int b = 0; b < NTB; ++b)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = row0 + 16 * rt + g + 8 * h, m = 8 * b + 2 * q + e;
          if (r >= R || m >= M) continue;
          const size_t o = static_cast<size_t>(m) * R + r;
          const float y0 = y[0][b][2 * h + e];
          if constexpr (MODE == MD_STORE) {
            out[o] = __float2bfloat16_rn(y0);
          } else if constexpr (MODE == MD_GATED) {
            const float y1 = y[NMAT - 1][b][2 * h + e];
            out[o] = __float2bfloat16_rn(s * act_f<ACT>(y0) * y1);
            if (o1) o1[o] = __float2bfloat16_rn(y0);
            if (o2) o2[o] = __float2bfloat16_rn(y1);
          } else {
            out[o] = __float2bfloat16_rn(s * act_f<ACT>(y0));
            if (o1) o1[o] = __float2bfloat16_rn(y0);
          }
        }
  }
}

// Warps per CTA: the most (up to the kernel's bound and the k groups) with
// which every CTA of the grid is resident at once.  Every CTA streams the
// same bytes, so with the whole grid resident they share HBM evenly and
// finish together; a second, partial wave would stream alone at the end.
// When no warp count fits the grid in one wave, two warps.
template <int ACT, int MODE, int NT>
int md_warps(int blocks, int ngroups) {
  static std::atomic<int> occ_cache[MD_MAX_WARPS + 1];  // CTAs per SM by warps, + 1 (0: unknown)
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 2;
  int best = 2;
  for (int w = 2; w <= md_max_threads<MODE>() / 32 && w <= ngroups; ++w) {
    int occ = occ_cache[w].load() - 1;
    if (occ < 0) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_decode_mma<ACT, MODE, NT>, 32 * w,
                                                        0) != cudaSuccess)
        return best;
      occ_cache[w].store(occ + 1);
    }
    if (static_cast<long long>(occ) * sms >= blocks) best = w;
  }
  return best;
}

template <int ACT, int MODE, int NT>
cudaError_t launch_md(const void* T, const void* W0, const void* W1, void* out, void* o1, void* o2,
                      int M, int R, int K, float s, cudaStream_t stream, bool pdl, int* status) {
  constexpr int rows = MD_ROWS * md_row_tiles<MODE, NT>();
  const int blocks = (R + rows - 1) / rows;
  const int ngroups = (K + MD_KG - 1) / MD_KG;
  const int warps = md_warps<ACT, MODE, NT>(blocks, ngroups);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(32 * warps, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_decode_mma<ACT, MODE, NT>,
                            static_cast<const __nv_bfloat16*>(T),
                            static_cast<const __nv_bfloat16*>(W0),
                            static_cast<const __nv_bfloat16*>(W1), static_cast<__nv_bfloat16*>(out),
                            static_cast<__nv_bfloat16*>(o1), static_cast<__nv_bfloat16*>(o2), M, R,
                            K, s, status);
}

template <int ACT, int MODE>
cudaError_t launch_md_nt(const void* T, const void* W0, const void* W1, void* out, void* o1,
                         void* o2, int M, int R, int K, float s, cudaStream_t stream, bool pdl,
                         int* status) {
  if (M <= 8)
    return launch_md<ACT, MODE, 8>(T, W0, W1, out, o1, o2, M, R, K, s, stream, pdl, status);
  return launch_md<ACT, MODE, 16>(T, W0, W1, out, o1, o2, M, R, K, s, stream, pdl, status);
}

}  // namespace

cudaError_t launch_decode_mma_act(const void* x, const void* Wg, const void* Wu, void* a, void* G,
                                  void* U, int M, int H, int I, int act, bool gated, float s,
                                  cudaStream_t stream, bool pdl, int* status) {
  if (M < 1 || M > DECODE_MMA_MAX_M) return cudaErrorInvalidValue;
  if (gated) {
    switch (act) {
      case ACT_RELU: return launch_md_nt<ACT_RELU, MD_GATED>(x, Wg, Wu, a, G, U, M, I, H, s, stream, pdl, status);
      case ACT_GELU_TANH: return launch_md_nt<ACT_GELU_TANH, MD_GATED>(x, Wg, Wu, a, G, U, M, I, H, s, stream, pdl, status);
      case ACT_SIGMOID: return launch_md_nt<ACT_SIGMOID, MD_GATED>(x, Wg, Wu, a, G, U, M, I, H, s, stream, pdl, status);
      default: return launch_md_nt<ACT_SILU, MD_GATED>(x, Wg, Wu, a, G, U, M, I, H, s, stream, pdl, status);
    }
  }
  switch (act) {
    case ACT_RELU: return launch_md_nt<ACT_RELU, MD_NONGATED>(x, Wg, nullptr, a, G, nullptr, M, I, H, s, stream, pdl, status);
    case ACT_GELU_TANH: return launch_md_nt<ACT_GELU_TANH, MD_NONGATED>(x, Wg, nullptr, a, G, nullptr, M, I, H, s, stream, pdl, status);
    default: return launch_md_nt<ACT_RELU_SQ, MD_NONGATED>(x, Wg, nullptr, a, G, nullptr, M, I, H, s, stream, pdl, status);
  }
}

cudaError_t launch_decode_mma_down(const void* a, const void* Wd, void* out, int M, int H, int I,
                                   cudaStream_t stream, bool pdl) {
  if (M < 1 || M > DECODE_MMA_MAX_M) return cudaErrorInvalidValue;
  return launch_md_nt<0, MD_STORE>(a, Wd, nullptr, out, nullptr, nullptr, M, H, I, 1.f, stream,
                                   pdl, nullptr);
}

}  // namespace mlpk
