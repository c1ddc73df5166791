/*
 * mlp.h -- C ABI of libmlp.so, the fused transformer MLP block on one GB300
 * (sm_103a) GPU, forward and backward.
 *
 * The operation (bf16 storage, fp32 accumulation, row-major everywhere):
 *
 *   g   = x Wg^T                    [M,I]   gate_proj(x)
 *   u   = x Wu^T                    [M,I]   up_proj(x)        (gated only)
 *   h   = gate_mult * act(g) * u    [M,I]   (non-gated: gate_mult * act(g))
 *   out = down_mult * h Wd^T        [M,H]   down_proj(h)
 *
 * with x [M,H], Wg/Wu [I,H] and Wd [H,I] in nn.Linear layout, no bias.
 * Sources:
 *   - flash-swiglu-mlp 0.4.2 README (PyPI METADATA), opening paragraph: the
 *     computed object down_proj(silu(gate_proj(x)) * up_proj(x)); section
 *     "Falcon H1 style models": the scaled form down_multiplier *
 *     down_proj(gate_multiplier * silu(gate_proj(x)) * up_proj(x)), both
 *     multipliers defaulting to 1.0; section "Supported configurations":
 *     no bias, contiguous [B,S,dim] input, rows 16-byte aligned (dim and
 *     hidden_dim multiples of 8 in bf16); section "Design notes": the
 *     backward in four stages with dG/dU written over G/U, the merged
 *     dW_g/dW_u GEMM and the single-accumulator dI; separate train and
 *     inference paths, the latter storing no G/U.
 *   - quack mlp.py (Tri Dao): MLP(activation=...) with the Activation
 *     literal (gelu_tanh_approx, relu_sq, swiglu, ...); mlp_func(x, weight1,
 *     weight2, activation, fuse_grad_accum, tuned, recompute);
 *     MLPRecomputeFunc (saves only x, recomputes preact = x W1^T in
 *     backward); _compute_weight_grad (fuse_grad_accum: W.grad += dout^T x
 *     in place, else a fresh gradient in the weight dtype); the
 *     needs_input_grad logic that skips unrequested gradients.
 *   - modded-nanogpt track_1_short/model/gpt.py, ReLUSqrdMLP:
 *     relu(x W1^T)^2 W2^T.
 *
 * Conventions shared by every entry point
 *   - Ownership: the caller allocates and owns every buffer (device memory);
 *     the library never allocates or frees device memory.  The only state it
 *     keeps is per-device properties and a cache of TMA descriptors keyed by
 *     (pointer, shape, box).
 *   - Streams: all work is enqueued on `stream` (a cudaStream_t, or NULL for
 *     the legacy default stream); nothing synchronises, except
 *     mlp_device_status.
 *   - Pointers marked bf16 hold __nv_bfloat16 values; every device pointer
 *     must be 16-byte aligned.  M, H, I > 0; H and I multiples of 8.
 *   - Return value: MLP_OK (0) or a negative mlp_status_t.  Arguments are
 *     validated before anything is enqueued; on a validation error nothing
 *     is enqueued and outputs are untouched.
 *   - Workspace: `ws` is caller-owned device scratch of at least
 *     mlp_workspace_size(p, mode) bytes, 256-byte aligned.  Its first 1 KB
 *     holds the device status word, the tile-scheduler counters and the
 *     one-launch gated forward's per-block counts; every call clears it on
 *     the stream before its kernels run (a decode weight stream, which uses
 *     no counters, clears only the status word, in its first kernel).
 *     Calls that share one workspace must be ordered (same stream, or
 *     synchronised).
 *   - Device-side errors (a bounded wait that expired) are recorded in the
 *     workspace status word; read it with mlp_device_status.
 *   - Determinism: two calls with the same inputs, problem, mode and tile
 *     policy write bitwise-identical outputs, except where the call splits
 *     a sum over K across work units (mlp_plan's out_split or wgrad_split
 *     above 1).  Those fp32 partial sums are added (in the workspace, or in
 *     the caller's fp32 weight gradients) in the order the units finish, so
 *     such outputs can differ in their last bits from one call to the next.
 *     The FP8 amax records are maxima and do not depend on that order.
 */
#ifndef MLP_GB300_H
#define MLP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLP_OK = 0,
  MLP_ERR_INVALID_ARG = -1,        /* null required pointer, M/H/I <= 0, bad enum, NULL problem */
  MLP_ERR_ALIGNMENT = -2,          /* H or I not a multiple of 8, or a pointer not 16-byte aligned */
  MLP_ERR_UNSUPPORTED = -3,        /* a combination the library does not implement */
  MLP_ERR_WORKSPACE_TOO_SMALL = -4,/* ws_bytes < mlp_workspace_size(p, mode) */
  MLP_ERR_CUDA = -5,               /* a CUDA runtime/driver call or a launch failed */
  MLP_ERR_TIMEOUT = -6             /* device side: a bounded wait expired (see mlp_device_status) */
} mlp_status_t;

/* Activation (quack mlp.py, the Activation literal).
 * Gated (a gate and an up weight, h = gate_mult * f(x Wg^T) * (x Wu^T)):
 *   SWIGLU f = silu(z) = z sigmoid(z)      REGLU f = relu(z) = max(z, 0)
 *   GEGLU  f = the tanh GELU below          GLU   f = sigmoid(z) = 1/(1+e^-z)
 * Non-gated (one fc1 weight, passed as Wg, and Wu must be NULL;
 * h = gate_mult * f(x Wg^T)):
 *   RELU_SQ f = relu(z)^2 (modded-nanogpt gpt.py, ReLUSqrdMLP)
 *   GELU_TANH f = 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))
 *   RELU f = max(z, 0)
 * The pages name reglu, geglu, glu and relu without formulas; these are the
 * plain readings (GLU: Dauphin et al. 2017; GLU variants: Shazeer 2020).
 * relu'(0) is taken as 0.  swiglu_oai, also named there, is not provided. */
typedef enum {
  MLP_ACT_SWIGLU = 0,
  MLP_ACT_RELU_SQ = 1,
  MLP_ACT_GELU_TANH = 2,
  MLP_ACT_RELU = 3,
  MLP_ACT_REGLU = 4,
  MLP_ACT_GEGLU = 5,
  MLP_ACT_GLU = 6
} mlp_act_t;

/* Problem description.  M = tokens (batch * sequence), H = hidden (model
 * dim), I = intermediate.  gate_mult and down_mult are the Falcon-H1
 * multipliers (1.0 for Llama-style MLPs). */
typedef struct {
  int M, H, I;
  int act;          /* mlp_act_t */
  float gate_mult;
  float down_mult;
} mlp_problem_t;

/* Workspace modes for mlp_workspace_size. */
typedef enum {
  MLP_MODE_FWD = 0,
  MLP_MODE_INFER = 1,
  MLP_MODE_BWD = 2,
  MLP_MODE_BWD_RECOMPUTE = 3,
  MLP_MODE_FP8_FWD = 4,  /* mlp_fp8_fwd: the control block + an e4m3 [M,I] postact */
  MLP_MODE_FP8_BWD = 5   /* mlp_fp8_bwd: the control block + e5m2 [M,H] and [M,I] codes */
} mlp_mode_t;

/* Bytes of workspace a call in `mode` needs for problem `p` (0 on invalid
 * arguments).  FWD/INFER/BWD: the control block plus one bf16 [M,I] buffer
 * (the postact); BWD_RECOMPUTE: plus the recomputed preacts, two bf16
 * [M,I] buffers when gated, one when not.  When the [M,H] output GEMM (the
 * down projection, or dx) has too few output tiles to fill the GPU, the GEMM
 * splits K and the workspace also holds one fp32 [M,H] partial-sum region:
 * decode-sized M (at most 32 tiles of 128 x 256 and K >= 1024), and for the
 * forward's down projection also at most 38 tiles of 256 x 256 (half of 76
 * CTA pairs: e.g. 384 or 512 tokens of a 4096-wide model), split so that
 * the units fill at least 80 % of their last wave.  The size depends on the
 * problem and mode only. */
size_t mlp_workspace_size(const mlp_problem_t* p, int mode);

/* Training forward (flash-swiglu-mlp README "Design notes", forward fusion;
 * quack mlp.py mlp_func with store_preact).
 *   x      bf16 [M,H]  in
 *   Wg     bf16 [I,H]  in   (non-gated: W1)
 *   Wu     bf16 [I,H]  in   (NULL when non-gated)
 *   Wd     bf16 [H,I]  in
 *   out    bf16 [M,H]  out
 *   G_save bf16 [M,I]  out, optional: the gate preact x Wg^T (non-gated: x W1^T)
 *   U_save bf16 [M,I]  out, optional: the up preact x Wu^T (NULL when non-gated)
 * Pass G_save/U_save as NULL for the recompute mode (save only x).  The
 * bf16 values written to `out` are bitwise identical to mlp_fwd_infer's.
 * With one to eight tokens (decode), unless a tile policy is set (below),
 * the forward streams the weights instead of running tensor-core GEMM
 * tiles (two kernels, no split-K region used): with three to eight tokens
 * each CTA owns 16 weight rows, its warps read them in 128-byte pieces per
 * row and accumulate the M dot products with the warp-level MMA (mma.sync,
 * bf16 in, fp32 accumulate) straight from the loaded registers; with one or
 * two tokens (M * max(H, I) * 2 <= 112 KiB) each warp reads whole weight
 * rows front to back and accumulates with fp32 fused multiply-adds on the
 * CUDA cores.  From nine tokens on, the tensor-core GEMMs with split-K. */
int mlp_fwd(const mlp_problem_t* p, const void* x, const void* Wg, const void* Wu,
            const void* Wd, void* out, void* G_save, void* U_save,
            void* ws, size_t ws_bytes, void* stream);

/* No-grad inference forward (flash-swiglu-mlp README, "inference path":
 * stores no G/U, only the transient postact in the workspace).
 * Arguments as in mlp_fwd. */
int mlp_fwd_infer(const mlp_problem_t* p, const void* x, const void* Wg, const void* Wu,
                  const void* Wd, void* out, void* ws, size_t ws_bytes, void* stream);

/* Backward from saved preacts (flash-swiglu-mlp README "Design notes",
 * the four backward stages; quack mlp.py backward of linear_gated_func /
 * gated_linear_func).
 *   dout  bf16 [M,H]  in   upstream gradient of out
 *   x, Wg, Wu, Wd     in   as in mlp_fwd
 *   G, U  bf16 [M,I]  in/out: in = the saved preacts from mlp_fwd; out =
 *                     overwritten with dG, dU (the gradients w.r.t. the
 *                     preacts), as flash-swiglu does to lower peak memory.
 *                     They are left untouched when dx, dWg and dWu are all
 *                     NULL.  U is NULL when non-gated.
 *   dx    bf16 [M,H]  out, or NULL to skip
 *   dWg, dWu [I,H], dWd [H,I]: each NULL to skip.  fuse_grad_accum = 0:
 *                     bf16, overwritten with the gradient.  fuse_grad_accum
 *                     = 1: fp32, dW += gradient in place (quack
 *                     _compute_weight_grad with fuse_grad_accum).
 * When only dWd is requested, the postact is rebuilt from G/U without the
 * activation derivative (quack MLPRecomputeFunc.backward, "only dW2 needed").
 * Streams: when dx and a weight gradient are both requested, the weight
 * gradients run on a second stream the library keeps per device, forked
 * from `stream` after the dgated GEMM and joined back into it before the
 * call returns (event record / wait, so the call stays capturable into a
 * CUDA graph once one direct backward call on the device has created that
 * stream).  Work enqueued on `stream` after the call sees every output.
 * Calls from several host threads or streams on one device are safe; a
 * capture and eager calls on one device should not overlap in time. */
int mlp_bwd(const mlp_problem_t* p, const void* dout, const void* x, const void* Wg,
            const void* Wu, const void* Wd, void* G, void* U, void* dx,
            void* dWg, void* dWu, void* dWd, int fuse_grad_accum,
            void* ws, size_t ws_bytes, void* stream);

/* Backward that saved only x (quack mlp.py MLPRecomputeFunc): recomputes
 * the preacts x Wg^T, x Wu^T into the workspace, then runs mlp_bwd's
 * stages.  Arguments as in mlp_bwd without G and U.  For the non-gated
 * activations, when dx, dWg or dWu is requested, the preact and dout Wd
 * are computed in the same output tile (two accumulators) and the epilogue
 * writes the postact and dP straight from them: the preact never reaches
 * memory. */
int mlp_bwd_recompute(const mlp_problem_t* p, const void* dout, const void* x,
                      const void* Wg, const void* Wu, const void* Wd, void* dx,
                      void* dWg, void* dWu, void* dWd, int fuse_grad_accum,
                      void* ws, size_t ws_bytes, void* stream);

/* ---- The MLP block with its neighbours ----
 * modded-nanogpt track_1_short/model/gpt.py, the layer loop's "process mlp":
 * `mlp_in = norm(x)`, the MLP, then
 * `x = scale_add(resid_lambdas_mlp[i], x, post_lambdas_mlp[i], mlp_out)`:
 *   y = resid_lambda * x + post_lambda * MLP(x / r),
 *   r = sqrt(mean_h x^2 + eps) per token (an RMS norm with no weight),
 * MLP as in mlp_fwd (activation, gate_mult, down_mult of `p`).  The norm is
 * fused into the gate/up GEMM (its epilogue scales the accumulator rows by
 * 1/r, computed by a small per-token kernel first), the residual add into
 * the down projection's epilogue.  Readings: the pages show the calls only;
 * norm is the plain RMS norm above, scale_add(a, x, b, y) = a x + b y. */
typedef struct {
  float resid_lambda;  /* scale of the residual stream x */
  float post_lambda;   /* scale of the MLP output (folded into down_mult) */
  float eps;           /* the RMS norm's epsilon (>= 0; F.rms_norm's default for bf16
                          inputs is 2^-7) */
} mlp_block_t;

/* Forward of the block.  Arguments as in mlp_fwd, plus
 *   b          the block's scalars (finite, eps >= 0), else MLP_ERR_INVALID_ARG
 *   y          bf16 [M,H] out; may be x itself (each element of x is read
 *              before its tile of y is written)
 *   G_save, U_save  the preacts of the normalised input, (x/r) Wg^T, (x/r) Wu^T
 *   rstd_save  fp32 [M] out, 16-byte aligned: 1/r per token (input of the backward)
 * Workspace: mlp_workspace_size(p, MLP_MODE_FWD). */
int mlp_block_fwd(const mlp_problem_t* p, const mlp_block_t* b, const void* x, const void* Wg,
                  const void* Wu, const void* Wd, void* y, void* G_save, void* U_save,
                  float* rstd_save, void* ws, size_t ws_bytes, void* stream);

/* Backward of the block from the saved preacts and rstd (as mlp_bwd):
 *   dy    bf16 [M,H] in: gradient of y
 *   dx    bf16 [M,H] out or NULL: resid_lambda dy plus the MLP's input
 *         gradient taken back through the RMS norm,
 *         dx = resid_lambda dy + (dn - n mean_h(dn n)) / r;  must not be x or dy
 *   dWg, dWu, dWd: as in mlp_bwd (gradients w.r.t. the weights of the MLP
 *         applied to x / r, with post_lambda dy as its output gradient)
 * The dgated / dact epilogue scales dG, dU (dP) by 1/r, so that dx's GEMM
 * and the weight gradients work on x itself; a per-token kernel then applies
 * the norm's projection term and adds the residual's gradient.
 * Workspace: mlp_workspace_size(p, MLP_MODE_BWD). */
int mlp_block_bwd(const mlp_problem_t* p, const mlp_block_t* b, const void* dy, const void* x,
                  const void* Wg, const void* Wu, const void* Wd, void* G, void* U,
                  const float* rstd, void* dx, void* dWg, void* dWu, void* dWd,
                  int fuse_grad_accum, void* ws, size_t ws_bytes, void* stream);

/* ---- FP8 forward and backward of the ReLU^2 MLP ----
 * modded-nanogpt gpt.py trains its ReLU^2 MLP with e4m3 operands and
 * dequant scales (a value is its e4m3 code times the scale; the constants
 * block above ReLUSqrdMLP and the _mlp_* buffers): the input's static scale
 * FP8_MLP_X_SCALE = 2^-4, amax/448 weight scales, and a delayed scale for
 * the ReLU^2 output (the last step's amax x 1.03 / 448) whose new amax the
 * kernels record.  The quantisation reading (the kernels are not on the
 * page): q = e4m3(fp32(v * fp32(1 / scale))), round to nearest even,
 * saturating at +-448.  The backward quantises the incoming gradient to
 * e5m2 with the static FP8_GRAD_SCALE = 2^-6 and the ReLU^2 derivative to
 * e5m2 with a delayed scale (the last step's amax x 1.25 / 57344), whose new
 * amax the kernels record; e5m2 saturates at +-57344. */

/* e4m3 codes of n bf16 values (n a multiple of 8; 16-byte aligned src and
 * dst): dst[i] = e4m3(src[i] * (1 / *scale)); with amax non-NULL, the
 * largest |src[i]| is atomically max-ed into *amax (which the caller zeroes
 * when it starts a new maximum).  scale and amax are device fp32 scalars. */
int mlp_fp8_quantize(const void* src, long long n, const float* scale, void* dst, float* amax,
                     void* stream);

/* Forward on e4m3 codes (p->act must be MLP_ACT_RELU_SQ, H and I multiples of 16):
 *   pre = (x8 W1_8^T) * sx * s1,   a = gate_mult * relu(pre)^2,
 *   a8  = e4m3(a * (1 / s_post)),  *amax_a = max(*amax_a, max |a|),
 *   out = down_mult * (a8 W2_8^T) * s_post * s2          (bf16 [M,H])
 *   x8 [M,H], W1_8 [I,H], W2_8 [H,I]: e4m3 codes (one byte each, row-major)
 *   scales: device fp32 {sx, s1, s2, s_post} (mlp_fp8_bwd's first four)
 *   a8_save: e4m3 [M,I] out, or NULL (then the workspace holds it)
 *   pre_save: bf16 [M,I] out (pre rounded to bf16, for mlp_fp8_bwd), or NULL
 *   amax_a: device fp32 scalar, or NULL
 * fc1 and the down projection are tcgen05 kind::f8f6f4 GEMMs (fp32
 * accumulation); the ReLU^2, its re-quantisation and amax run in fc1's
 * epilogue.  Workspace: mlp_workspace_size(p, MLP_MODE_FP8_FWD). */
int mlp_fp8_fwd(const mlp_problem_t* p, const void* x8, const void* W1_8, const void* W2_8,
                const float* scales, void* out, void* a8_save, void* pre_save, float* amax_a,
                void* ws, size_t ws_bytes, void* stream);

/* Backward on 8-bit codes, the chain rule through the forward above with
 * straight-through quantisations (p->act MLP_ACT_RELU_SQ, H and I multiples of 16):
 *   dout8 = e5m2(dout * (1 / sg)),
 *   dpre  = gate_mult * down_mult * (dout8 W2_8) * sg * s2 * 2 relu(pre),
 *   dP8   = e5m2(dpre * (1 / s_dpre)),  *amax_dpre = max(*amax_dpre, max |dpre|),
 *   dx    = (dP8 W1_8) * s_dpre * s1                          (bf16 [M,H])
 *   dW1   = (dP8^T x8) * s_dpre * sx                          (bf16 [I,H])
 *   dW2   = down_mult * (dout8^T a8) * sg * s_post            (bf16 [H,I])
 *   dout: bf16 [M,H];  pre: the forward's pre_save (bf16 [M,I]), or NULL: then the
 *         derivative GEMM recomputes the preact in each output tile from x8 and
 *         W1_8 (a second accumulator, the forward's own fp32 sums) and forms
 *         2 relu(pre) from it rounded to bf16 as the saved path does, so the
 *         codes, dx, dW1 and dW2 are the same as with the forward's pre_save
 *         (the forward then need not write it);  a8: the forward's e4m3 postact
 *   x8, W1_8, W2_8: the forward's e4m3 codes
 *   scales: device fp32 {sx, s1, s2, s_post, sg, s_dpre}
 *   dx, dW1, dW2: outputs, each NULL when not wanted (then its operands may be NULL)
 *   amax_dpre: device fp32 scalar, or NULL
 * All three GEMMs are tcgen05 kind::f8f6f4 (e5m2 x e4m3, fp32 accumulation)
 * and read W1_8, W2_8, x8 and a8 in their row-major layout (MN-major
 * operands): no transposed copies.  dx and the grouped weight gradients may
 * run on a second stream, joined before the call returns.  Workspace:
 * mlp_workspace_size(p, MLP_MODE_FP8_BWD). */
int mlp_fp8_bwd(const mlp_problem_t* p, const void* dout, const void* x8, const void* W1_8,
                const void* W2_8, const void* pre, const void* a8, const float* scales, void* dx,
                void* dW1, void* dW2, float* amax_dpre, void* ws, size_t ws_bytes, void* stream);

/* Delayed-scale refresh (modded-nanogpt gpt.py, _refresh_delayed_scale, as
 * _quantize_mlp_weights_and_scales calls it after every optimizer step): for
 * each of n slots, a = the largest of the slot's `width` recorded amax values
 * (amax is fp32 [n, width], row-major; a NaN or an infinity among them makes
 * a = 0), clamped to at most 1e12; if a > 0 the slot's scale becomes
 * max(a * gain, floor), else it keeps its value; then the slot's amax values
 * are set to 0.  The page's two uses, with the amax that mlp_fp8_fwd and
 * mlp_fp8_bwd record:
 *   s_post (scales[3]): amax_a,    gain = 1.03 / 448,    floor = 1e-6
 *   s_dpre (scales[5]): amax_dpre, gain = 1.25 / 57344,  floor = 1e-12
 * One small kernel on `stream`: a training loop can keep the refresh on the
 * device (and inside a captured CUDA graph) instead of reading the amax on
 * the host.  amax and scale: device fp32, 4-byte aligned, not overlapping.
 * n = 0 enqueues nothing; n < 0, width < 1, a NULL pointer or a non-finite
 * gain or floor is MLP_ERR_INVALID_ARG. */
int mlp_fp8_refresh_scales(float* amax, float* scale, int n, int width, float gain, float floor,
                           void* stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* mlp_status_string(int status);

/* Synchronises `stream`, then returns the device status word of the last
 * call that used workspace `ws` (MLP_OK or MLP_ERR_TIMEOUT), or
 * MLP_ERR_CUDA if the synchronisation or the copy failed. */
int mlp_device_status(const void* ws, void* stream);

/* Library version, e.g. "0.1.0". */
const char* mlp_version(void);

/* ---- Inference forward without a caller workspace (no counterpart on the
 * pages: an addition of this library) ----
 * For callers that may not allocate device memory when they run the MLP
 * (for example a C runtime whose device memory is planned once at start-up,
 * or a serving loop that must not call cudaMalloc because it synchronises
 * the device and has no caching allocator to draw from).  Same arguments and
 * results as mlp_fwd_infer, minus the workspace: the scratch is a fixed
 * device array of MLP_NOALLOC_SCRATCH_BYTES inside the library, present on
 * every GPU that loads the library until the process exits.
 *   - Returns MLP_ERR_WORKSPACE_TOO_SMALL, enqueueing nothing, when
 *     mlp_workspace_size(p, MLP_MODE_INFER) exceeds
 *     MLP_NOALLOC_SCRATCH_BYTES (about M * I <= 8.3 million elements).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress, with that device current), so the address stays
 *     right after a device reset; the first lookup on a device may load the
 *     library's device code, so make the first call before any stream
 *     capture.
 *   - All calls share the one array: it keeps the last call's contents, and
 *     each call clears the parts that must start at zero.  Calls whose work
 *     overlaps on the GPU (different streams, or without ordering) race on
 *     it; order them, e.g. on one stream. */
#define MLP_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int mlp_fwd_infer_noalloc(const mlp_problem_t* p, const void* x, const void* Wg, const void* Wu,
                          const void* Wd, void* out, void* stream);

/* The device status word of mlp_fwd_infer_noalloc's scratch on the current
 * device, as mlp_device_status reads a workspace's: synchronises `stream`,
 * then returns MLP_OK, or MLP_ERR_TIMEOUT when a bounded wait of the last
 * call expired (its output is then incomplete), or MLP_ERR_CUDA.  The word
 * is cleared at the start of every call. */
int mlp_noalloc_status(void* stream);

/* ---- Launch plan (introspection; no counterpart on the pages) ----
 * What one call in `mode` launches for problem `p` on the current device,
 * with every gradient requested (the backward modes) and the current tile
 * policy.  The split-K factors depend on the device's SM count. */
typedef struct {
  int decode;           /* the forward streams the weights (1-8 tokens; up to 16 when forced):
                           2 with the warp-level MMA, 1 on the CUDA cores; 0: GEMM tiles */
  int fused_forward;    /* 1: the gated forward's gate/up and down GEMMs are one launch */
  int cta_group;        /* CTA-group size (1 or 2) of the GEMMs over token rows */
  int out_split;        /* split-K factor of the [M,H] output GEMM (down projection, or dx) */
  int wgrad_cta_group;  /* CTA-group size of the weight-gradient launch */
  int wgrad_split;      /* split-K factor of the weight-gradient launch (> 1 only when
                           fuse_grad_accum: the splits meet by fp32 atomic adds in dW) */
} mlp_plan_t;
/* Fills *plan; MLP_ERR_INVALID_ARG for an invalid problem, mode or a NULL
 * plan, MLP_ERR_CUDA when no device can be queried.  Enqueues nothing. */
int mlp_plan(const mlp_problem_t* p, int mode, int fuse_grad_accum, mlp_plan_t* plan);

/* Tile policy (a tuning and testing knob; no counterpart on the pages):
 * 0 = automatic (default): GEMMs whose output has more than 128 rows use
 *     256 x 256 tiles computed by a CTA pair (tcgen05 cta_group::2), the
 *     others 128 x 256 tiles on one CTA;
 * 1 = always single-CTA tiles;  2 = always CTA-pair tiles;
 * 3 = as 0, but the gated forward's gate/up and down GEMMs run as two
 *     launches (policy 0 runs them as one; see MLP_KERNEL_FWD_FUSED).
 * Policies 1 and 2 also keep forwards of one to eight tokens on the
 * tensor-core GEMMs (policies 0 and 3 stream their weights, above).
 * Process-wide; returns MLP_ERR_INVALID_ARG for other values.  Results of
 * the two tile shapes agree to rounding (same fp32 accumulation order). */
int mlp_set_tile_policy(int policy);

/* ---- Failure-detection hooks (testing; no counterpart on the pages) ----
 * Every device-side wait of the kernels is bounded; when one expires the
 * kernel records MLP_ERR_TIMEOUT in the workspace status word, stops its
 * work and returns, leaving the CUDA context usable.
 * mlp_set_wait_timeout_ms sets the bound for later calls (0 = default:
 * the MLP_WAIT_TIMEOUT_MS environment variable, else 2000 ms).
 * mlp_debug_set_flags(MLP_DEBUG_NO_WORK) makes the kernels' tile schedulers
 * publish no work, so the bounded waits of every later call expire (a test
 * of the timeout path that issues no copy and no MMA); 0 restores normal
 * operation.  The decode flags pick one of the two weight streams of the
 * decode-sized forward (mlp_fwd): MLP_DEBUG_DECODE_FMA the CUDA-core one for
 * one to four tokens whose token rows fit a CTA's shared memory
 * (M * max(H, I) * 2 <= 112 KiB), MLP_DEBUG_DECODE_MMA the warp-MMA one for
 * one to sixteen tokens (it wins when both are set).  Flags may be
 * combined; both settings are process-wide. */
#define MLP_DEBUG_NO_WORK 1
#define MLP_DEBUG_DECODE_FMA 2
#define MLP_DEBUG_DECODE_MMA 4
int mlp_set_wait_timeout_ms(unsigned int ms);
int mlp_debug_set_flags(int flags);

/* Contention hook (testing): enqueues on `stream` one kernel of `ctas` CTAs
 * that each take enough shared memory to keep any GEMM CTA of this library
 * off their SM, and return after `us` microseconds (read from the GPU's
 * global timer; at most 10 s).  Work launched meanwhile on other streams
 * runs on the SMs left free: this tests that the kernels finish correctly
 * when only part of their grid is resident.  The kernel reads and writes no
 * memory and waits on nothing but the timer.  ctas in 1..65535, else
 * MLP_ERR_INVALID_ARG. */
int mlp_debug_hold_sms(int ctas, unsigned int us, void* stream);

/* ---- Tracing (timing support; no counterpart on the pages) ----
 * With tracing on, every kernel launch of the calls above is bracketed by
 * a pair of CUDA events recorded on the call's stream (this may keep
 * consecutive kernels from overlapping through programmatic dependent
 * launch), and the backward runs its weight-gradient GEMMs after dx on the
 * call's stream instead of beside it on the library's second stream, so
 * that each traced duration is one kernel's own.  Kernel tags: */
typedef enum {
  MLP_KERNEL_GATE_UP = 0,  /* gate/up (or fc1) GEMM with the activation epilogue */
  MLP_KERNEL_DOWN = 1,     /* down projection GEMM */
  MLP_KERNEL_DGATED = 2,   /* dout Wd GEMM with the dgated / dact epilogue */
  MLP_KERNEL_DX = 3,       /* dx GEMM */
  MLP_KERNEL_WGRAD = 4,    /* grouped weight-gradient GEMMs */
  MLP_KERNEL_POSTACT = 5,  /* elementwise postact rebuild (dWd-only backward) */
  MLP_KERNEL_CONVERT = 6,  /* fp32 -> bf16 of a split-K output (decode-sized M) */
  MLP_KERNEL_DACT_RECOMPUTE = 7, /* non-gated recompute: x W1^T and dout Wd in one tile,
                                    epilogue postact and dP */
  MLP_KERNEL_RSTD = 8,          /* the block's per-token RMS-norm scale */
  MLP_KERNEL_RMSNORM_BWD = 9,   /* the block's RMS-norm derivative and residual gradient */
  MLP_KERNEL_QUANT = 10,        /* bf16 -> e4m3 / e5m2 quantisation */
  MLP_KERNEL_FWD_FUSED = 11,    /* the gated forward's gate/up and down GEMMs in one launch
                                   (CTA-pair tiles, M <= 32768): a down tile starts once the
                                   postact of its 256 rows is stored */
  MLP_KERNEL_REFRESH = 12       /* the FP8 delayed-scale refresh */
} mlp_kernel_t;

/* on != 0 starts recording, 0 stops (records already taken are kept). */
int mlp_trace_enable(int on);

/* Waits for the recorded events, writes up to `capacity` (tag, ms) pairs
 * in launch order into host arrays `tags` and `ms`, frees all records, and
 * returns the number written (or MLP_ERR_CUDA). */
int mlp_trace_read(int* tags, float* ms, int capacity);

/* Static name of a kernel tag ("dgated", ...). */
const char* mlp_kernel_name(int tag);

#ifdef __cplusplus
}
#endif
#endif /* MLP_GB300_H */
