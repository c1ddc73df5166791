// gemm_params.h -- launch parameters shared by the host code and the
// persistent tcgen05 GEMM kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mlpk {

// Tile: (128 x CTA-group size) x (MMA N = 256) x BK, bf16 operands, fp32
// accumulators; each CTA owns BM = 128 accumulator rows.
constexpr int BM = 128;
constexpr int MMA_N = 256;
constexpr int BK = 64;
constexpr int SCHED_SLOTS = 8;
constexpr int NUM_EPI_WARPS = 8;                // two per TMEM lane quadrant (column halves)
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;  // producer, MMA, epilogue warps
constexpr int TMEM_COLS = 512;                  // two 256-column accumulators
constexpr int MAX_PROBS = 3;

// L2 cache policies of the operand loads (Prob::l2a, l2b).  The launches
// mark the operand that many tiles re-read evict-last and, where the other
// streams past once per tile column, that one evict-first: same-call A/B on
// the bf16 training steps, 2.3-3.0 % faster (SwiGLU shapes), 0.6 % (ReLU^2).
enum L2Policy : int { L2_NORMAL = 0, L2_EVICT_LAST = 1, L2_EVICT_FIRST = 2 };
constexpr int MAX_MAPS = 12;

// What the epilogue does with the accumulator tile.
enum Epi : int {
  EPI_GATED_FWD = 0,   // acc = [g | u] (128 + 128 cols): a = s*act(g)*u; optional G, U stores
  EPI_ACT_FWD = 1,     // acc = p (256 cols): a = s*act(p); optional P store
  EPI_DGATED = 2,      // acc = dout*Wd: dG = s*acc*u*act'(g), dU = s*acc*act(g), a = s*act(g)*u
  EPI_DACT = 3,        // acc = dout*Wd: dP = s*acc*act'(p), a = s*act(p)
  EPI_STORE_BF16 = 4,  // D = bf16(acc)
  EPI_ACCUM_F32 = 5,   // D += acc (fp32, atomic add; split-K safe)
  // non-gated backward with the preact recomputed in the same tile:
  // segment 0 acc = p = x W1^T (accumulator 0), segment 1 acc = dh = dout Wd
  // (accumulator 1): a = s*act(p), dP = s*dh*act'(p)
  EPI_DACT_RECOMP = 6,
  // 8-bit operands (tcgen05 kind::f8f6f4; e4m3 or e5m2 per operand, Params::f8_formats)
  // with the problem's dequant factor deq = mult * *sa * *sb:
  EPI_ACT_FWD_F8 = 7,     // pre = deq'*acc (deq' = *sa * *sb), a = mult*relu(pre)^2 ->
                          // e4m3(a / *sq) (map 0), optional bf16 pre (map 1), amax|a| -> *amax
  EPI_STORE_BF16_F8 = 8,  // D = bf16(deq * acc)
  EPI_DGRAD_F8 = 9,       // dpre = deq*acc*2*relu(P) (in0 = P, bf16) -> e5m2(dpre / *sq)
                          // (map 0), amax|dpre| -> *amax
  // The gated forward in one launch: problem 0 is the gate/up GEMM with the
  // EPI_GATED_FWD epilogue, problem 1 the down projection with the
  // EPI_STORE_BF16 epilogue, reading problem 0's postact.  A down unit of a
  // 256-row block starts once every gate/up tile of that block is stored
  // (Params::dep), so the down tiles fill the SMs the gate/up tail leaves idle.
  EPI_FWD_FUSED = 10,
  // The 8-bit derivative with the preact recomputed in the same tile
  // (nothing saved by the forward): segment 0 acc = x8 W1_8^T (accumulator
  // 0, both e4m3, B K-major), segment 1 acc = dout8 W2_8 (accumulator 1,
  // e5m2 x e4m3, B MN-major).  dd = bf16(2 relu(deq0 * acc0)) is held per
  // thread between the two, then dpre = mult * deq * acc1 * dd ->
  // e5m2(dpre / *sq) (map 0), amax|dpre| -> *amax.  dd is the value the
  // saved-preact path forms from the preact it stores in bf16, so both give
  // the same codes.
  EPI_DGRAD_F8_RECOMP = 11
};

__host__ __device__ constexpr bool is_f8(int epi) {
  return epi == EPI_ACT_FWD_F8 || epi == EPI_STORE_BF16_F8 || epi == EPI_DGRAD_F8 ||
         epi == EPI_DGRAD_F8_RECOMP;
}
// Epilogues whose tiles accumulate two K segments into the two accumulators
// (segment 0's B K-major, segment 1's B MN-major).
__host__ __device__ constexpr bool is_recomp(int epi) {
  return epi == EPI_DACT_RECOMP || epi == EPI_DGRAD_F8_RECOMP;
}
// 8-bit operand formats of Params::f8_formats (the kind::f8f6f4 type codes)
constexpr int F8_E4M3 = 0, F8_E5M2 = 1;

// The function applied to the gate (gated MLPs) or to the preact (non-gated).
enum Act : int { ACT_SILU = 0, ACT_RELU_SQ = 1, ACT_GELU_TANH = 2, ACT_RELU = 3, ACT_SIGMOID = 4 };

// One GEMM D[M,N] = sum_k A[m,k] B[n,k] of a (possibly grouped) launch.
struct Prob {
  int M, N;               // output rows / columns
  int kb0, kb1;           // k-blocks of K-segment 0 and 1 (kb1 = 0: one segment)
  int tiles_m, tiles_n;   // output tiles (tile N = 128 for a gated forward, else 256)
  int ksplit, kper;       // split-K factor, k-blocks per split
  int unit_begin, units;  // this problem's slice of the global work-unit range
  int mapA0, mapB0;       // tensor maps of segment 0
  int mapA1, mapB1;       // segment 1 (EPI_GATED_FWD: mapB1 = the up weight;
                          // EPI_DACT_RECOMP: B is K-major in segment 0, MN-major in 1)
  int ld;                 // row pitch (elements) of the epilogue's outputs and inputs
  int mapI0, mapI1;       // derivative epilogues: maps of in0 / in1 with boxes {256, 128}
                          // whose tiles the producer prefetches into L2 (-1: none)
  int mapE;               // EPI_DGRAD_F8: map of in0 with the epilogue warps' 32 x 32 bf16
                          // boxes (64-byte swizzle), loaded by TMA (-1: plain loads)
  int mapO[3];            // tensor maps of the epilogue's outputs (-1: output not written)
  void* out0;
  void* out1;
  void* out2;
  const void* in0;
  const void* in1;
  // the MLP block's neighbours (0 / nullptr: none):
  const float* rstd;      // per output row: gate/up accumulators (activation forward) and
                          // dG, dU / dP (derivative epilogues) are multiplied by rstd[row]
  float alpha;            // EPI_STORE_BF16 with in0 = residual [M, ld]: D = alpha*in0 + acc
  int group_m;            // L2 raster group of this problem (0: Params::group_m)
  int l2a, l2b;           // L2 policy of the A / B operand loads (L2Policy)
  // 8-bit epilogues: dequant factor mult * *sa * *sb; *sq the scale of an 8-bit output
  const float* sa;
  const float* sb;
  const float* sq;
  float mult;
  float* amax;            // running max of |the quantised output| (atomic; may be null)
  // EPI_DGRAD_F8_RECOMP: the recomputed preact's dequant scales (sx, s1)
  const float* sp0;
  const float* sp1;
};

struct Params {  // 64-byte aligned through CUtensorMap
  CUtensorMap maps[MAX_MAPS];
  Prob prob[MAX_PROBS];
  int nprob;
  int total_units;
  int act;
  int group_m;            // L2 raster: tiles are visited in groups of group_m tile rows
  float scale;            // gate_mult * down_mult (activation epilogues)
  int f8_formats;         // 8-bit MMAs: A's format (bits 0-2) and B's (bits 3-5), F8_*
  int f8_formats0;        // EPI_DGRAD_F8_RECOMP: the formats of K segment 0 (f8_formats: segment 1)
  int debug_flags;        // MLP_DEBUG_* (testing only; 0 in normal use)
  int a_tx_bytes;         // bytes one CTA's A boxes bring per k-block (K-major A: rows x 128 B)
  int nmaps;              // tensor maps in use
  int dep_target;         // EPI_FWD_FUSED: dep count of a complete 256-row block
  int* counter;           // dynamic tile scheduler counter, zero at launch
  int* status;            // device status word (MLP_ERR_TIMEOUT on a bounded-wait expiry)
  int* dep;               // EPI_FWD_FUSED: per 256-row block, the gate/up epilogue warps whose
                          // stores have completed (one count per warp and tile; zero at launch)
  unsigned long long timeout_ns;
};

// Host-side launcher and co-residency query, explicitly instantiated in the
// kernel translation units.  CG = CTA-group size (1: single CTA, 2: CTA
// pair with tcgen05 cta_group::2); `grid` is in CTAs (a multiple of CG).
// ACT is the activation of the activation epilogues (0 for the others).
template <int EPI, bool A_MN, bool B_MN, int CG, int ACT>
cudaError_t launch_gemm(const Params& p, int grid, cudaStream_t stream, bool pdl);
template <int EPI, bool A_MN, bool B_MN, int CG, int ACT>
int max_groups();

// Elementwise postact a = s*act(G)*U (U == nullptr: non-gated), n elements;
// `act` is a device activation (Act).
cudaError_t launch_postact(const void* G, const void* U, void* a, long long n, int act,
                           float scale, cudaStream_t stream, bool pdl);

// fp32 -> bf16 (round to nearest even), n elements (a multiple of 8); with
// `resid` (bf16, n elements) the result is src + alpha * resid.
cudaError_t launch_f32_to_bf16(const float* src, void* dst, long long n, cudaStream_t stream,
                               bool pdl, const void* resid = nullptr, float alpha = 0.f);

// 8-bit codes q = f8(fp32(src * fp32(1 / *scale))) of n bf16 values, f8 = e4m3
// (fmt F8_E4M3) or e5m2 (F8_E5M2), saturating, round to nearest even; with
// `amax`, atomic max of |src| into *amax.
cudaError_t launch_quant_f8(const void* src, long long n, const float* scale, void* dst,
                            float* amax, int fmt, cudaStream_t stream, bool pdl);

// The delayed-scale refresh of n slots (amax fp32 [n, width], scale fp32 [n]):
// scale = max(a * gain, floor) where a = the slot's finite amax (> 0), amax
// cleared.
cudaError_t launch_refresh_scales(float* amax, float* scale, int n, int width, float gain,
                                  float floor_v, cudaStream_t stream, bool pdl);

// Testing: `ctas` CTAs, each holding HOLD_SMEM_BYTES of shared memory (so no
// GEMM CTA shares its SM), return after `ns` nanoseconds of the global timer.
constexpr int HOLD_SMEM_BYTES = 120 * 1024;
cudaError_t launch_hold(int ctas, unsigned long long ns, cudaStream_t stream);

// Decode-sized forward (M <= DECODE_MAX_M) on the CUDA cores: the gate/up
// (or fc1) pass with its activation (a, and G/U or P when given), and the
// down projection out = a Wd^T.  `act` is a device activation (Act).  Each
// CTA stages the M token rows of its K (H, then I) whole in shared memory:
// M * K * 2 <= DECODE_MAX_TOKEN_BYTES.  The gate/up pass, the first kernel
// of its call, also clears the call's status word (`status`, may be null).
constexpr int DECODE_MAX_M = 4;
// (112 KiB: four token rows of a 14336-wide intermediate; two such CTAs,
// with the 1 KiB each reserves, fit an SM's 228 KiB of shared memory)
constexpr int DECODE_MAX_TOKEN_BYTES = 112 * 1024;
cudaError_t launch_decode_act(const void* x, const void* Wg, const void* Wu, void* a, void* G,
                              void* U, int M, int H, int I, int act, bool gated, float s,
                              cudaStream_t stream, bool pdl, int* status);
cudaError_t launch_decode_down(const void* a, const void* Wd, void* out, int M, int H, int I,
                               cudaStream_t stream, bool pdl);

// Decode-sized forward (M <= DECODE_MMA_MAX_M) on the warp-level MMA: the
// same two passes and epilogues as above, the dot products as mma.sync
// m16n8k16 (bf16 in, fp32 accumulate) fed straight from 16-byte loads; the
// token rows are read through the caches, so K is not limited.
constexpr int DECODE_MMA_MAX_M = 16;
// Tokens up to which the library takes the warp-MMA stream by itself: with
// 9-16 tokens (two 8-token blocks) the stream measured no faster than the
// tensor-core GEMMs (74.9-75.9 against 74.0-75.9 us on Llama-3-8B's
// weights; 81-83 us before its down pass took two row tiles per warp)
constexpr int DECODE_MMA_AUTO_M = 8;
cudaError_t launch_decode_mma_act(const void* x, const void* Wg, const void* Wu, void* a, void* G,
                                  void* U, int M, int H, int I, int act, bool gated, float s,
                                  cudaStream_t stream, bool pdl, int* status);
cudaError_t launch_decode_mma_down(const void* a, const void* Wd, void* out, int M, int H, int I,
                                   cudaStream_t stream, bool pdl);

// Per-token RMS-norm scale rstd[m] = 1 / sqrt(mean_h x^2 + eps), x bf16 [M, H].
cudaError_t launch_rstd(const void* x, float* rstd, int M, int H, float eps, cudaStream_t stream,
                        bool pdl);

// In place over dx (holding D = dn * rstd): dx = alpha dy + D - (rstd^2 / H) (sum_h D x) x.
cudaError_t launch_rmsnorm_bwd(void* dx, const void* x, const void* dy, const float* rstd, int M,
                               int H, float alpha, cudaStream_t stream, bool pdl);

}  // namespace mlpk
