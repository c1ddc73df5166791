// mlp_api.cu -- the C ABI of libmlp.so (declared in include/mlp.h):
// argument validation, workspace layout, TMA descriptor construction (with
// a cache keyed by pointer/shape/box), and the launch sequences of the
// forward, inference and backward passes.
//
// Launch sequences (every GEMM is the persistent tcgen05 kernel of gemm.cuh):
//   mlp_fwd / mlp_fwd_infer
//     1. gate/up GEMM, epilogue a = s*act(g)*u (+ G, U stores in training)
//     2. down GEMM  out = a Wd^T            (s = gate_mult*down_mult is folded into a)
//   mlp_bwd (the four stages of the flash-swiglu-mlp README, "Design notes")
//     1. dgated GEMM  dout Wd  (K = H), epilogue dG, dU over G, U and the postact a
//     2. dx GEMM      [dG|dU] [Wg;Wu]  (K = 2I, one accumulator)
//     3. one grouped launch of the weight gradients dWg = dG^T x, dWu = dU^T x,
//        dWd = dout^T a  (K = M), bf16 store or fp32 in-place accumulation,
//        on a second stream beside stage 2 when both are requested
//   mlp_bwd_recompute
//     0. gate/up GEMM storing only G, U into the workspace, then as mlp_bwd.
//     Non-gated with dx/dWg requested: stages 0 and 1 are one kernel whose
//     tiles accumulate p = x W1^T and dh = dout Wd in the two accumulators;
//     its epilogue writes the postact a and dP (p never reaches memory).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "gemm_params.h"
#include "mlp.h"

using namespace mlpk;

namespace {

// The workspace's control block (zeroed by every call): the status word
// (int 0), the tile-scheduler counters (ints 16..127) and the fused
// forward's per-block counts (ints 128..255).
constexpr size_t CTRL_BYTES = 1024;
constexpr int COUNTER_BASE = 16;
constexpr int MAX_COUNTERS = 112;
constexpr int DEP_BASE = 128;
constexpr int MAX_DEP_BLOCKS = 128;  // 256-row blocks of a fused forward: M <= 32768

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encode_fn_ok() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

struct MapKey {
  const void* ptr;
  uint64_t inner, outer, stride;
  uint32_t box0, box1;
  int dtype, swizzle;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && inner == o.inner && outer == o.outer && stride == o.stride &&
           box0 == o.box0 && box1 == o.box1 && dtype == o.dtype && swizzle == o.swizzle;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    size_t h = reinterpret_cast<size_t>(k.ptr);
    h = h * 1000003u ^ k.inner;
    h = h * 1000003u ^ k.outer;
    h = h * 1000003u ^ k.stride;
    h = h * 1000003u ^ (static_cast<size_t>(k.box0) << 16 | k.box1);
    h = h * 1000003u ^ (static_cast<size_t>(k.dtype) << 8 | static_cast<size_t>(k.swizzle));
    return h;
  }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;

// 2-D tensor map over a row-major [outer, inner] array with row pitch `pitch`
// elements, box {box0 (inner), box1 (outer)}; out-of-bounds elements read as
// zero and are not written.  bf16 operands use the 128-byte swizzle; the
// epilogue's 32 x 32 output boxes use the 64-byte (bf16) or 128-byte (fp32)
// swizzle of the staging buffers.
// dtype: 0 bf16, 1 fp32, 2 e4m3 bytes (uint8).
bool make_map(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer, uint64_t pitch,
              uint32_t box0, uint32_t box1, int dtype = 0,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  MapKey key{ptr, inner, outer, pitch, box0, box1, dtype, static_cast<int>(swz)};
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_map_cache.find(key);
    if (it != g_map_cache.end()) {
      *out = it->second;
      return true;
    }
  }
  if (!encode_fn_ok()) return false;
  const uint64_t esize = dtype == 1 ? 4 : (dtype == 2 ? 1 : 2);
  const CUtensorMapDataType dt = dtype == 1   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                              : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch * esize};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  CUresult r = g_encode(&m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lk(g_map_mu);
  if (g_map_cache.size() > 4096) g_map_cache.clear();
  g_map_cache.emplace(key, m);
  *out = m;
  return true;
}

// ------------------------------------------------------------ device info
int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

std::atomic<unsigned long long> g_wait_ms{0};  // 0: the default below
std::atomic<int> g_debug_flags{0};

unsigned long long wait_limit_ns() {
  static unsigned long long env_ms = [] {
    const char* e = std::getenv("MLP_WAIT_TIMEOUT_MS");
    return e ? std::strtoull(e, nullptr, 10) : 0ull;
  }();
  unsigned long long ms = g_wait_ms.load();
  if (ms == 0) ms = env_ms;
  if (ms == 0) ms = 2000;  // 2 s: far above any legitimate wait (tiles take microseconds)
  return ms * 1000000ull;
}

// ------------------------------------------------------------ launch builder
// Operand roles: a K-major operand [rows, K] is loaded with boxes
// {64, rows-per-box}; an MN-major operand [K, MN] with boxes {64, 64}.
// The device activation (Act) an ABI activation applies to the gate or preact.
int device_act(int act) {
  switch (act) {
    case MLP_ACT_SWIGLU: return ACT_SILU;
    case MLP_ACT_RELU_SQ: return ACT_RELU_SQ;
    case MLP_ACT_GELU_TANH: return ACT_GELU_TANH;
    case MLP_ACT_RELU: return ACT_RELU;
    case MLP_ACT_REGLU: return ACT_RELU;
    case MLP_ACT_GEGLU: return ACT_GELU_TANH;
    case MLP_ACT_GLU: return ACT_SIGMOID;
    default: return ACT_SILU;
  }
}

// 0 auto, 1 single-CTA tiles, 2 CTA-pair tiles, 3 auto with the gated
// forward's two GEMMs as separate launches
std::atomic<int> g_tile_policy{0};

// Which kernels a forward of few tokens streams its weights with (unless a
// tile policy forces the tensor-core GEMMs): 1, the CUDA-core stream, for
// one or two tokens whose rows fit a CTA's shared memory (measured 3-6 %
// faster than the warp-MMA stream there); 2, the warp-MMA stream, for the
// others up to DECODE_MMA_AUTO_M tokens; 0, the tensor-core GEMMs.  The
// testing flags force one stream: MLP_DEBUG_DECODE_FMA the CUDA-core one
// (up to four tokens that fit), MLP_DEBUG_DECODE_MMA the warp-MMA one (up to
// DECODE_MMA_MAX_M tokens).
int decode_kernel(const mlp_problem_t* p) {
  const int pol = g_tile_policy.load();
  if ((pol != 0 && pol != 3) || p->M > DECODE_MMA_MAX_M) return 0;
  const int flags = g_debug_flags.load();
  if (flags & MLP_DEBUG_DECODE_MMA) return 2;
  const long long k = p->H > p->I ? p->H : p->I;
  const bool fma_fits = p->M <= DECODE_MAX_M && (long long)p->M * k * 2 <= DECODE_MAX_TOKEN_BYTES;
  if (fma_fits && (p->M <= 2 || (flags & MLP_DEBUG_DECODE_FMA))) return 1;
  return p->M <= DECODE_MMA_AUTO_M ? 2 : 0;
}

// CTA-group size for a GEMM whose output has `rows` rows: pairs (256-row
// tiles) unless the output fits one 128-row tile.
int pick_cg(int rows) {
  const int pol = g_tile_policy.load();
  if (pol == 1 || pol == 2) return pol;
  return rows > BM ? 2 : 1;
}

struct Gemm {
  Params p;
  int nmaps = 0;
  int cg = 1;
  bool ok = true;
  Gemm(const mlp_problem_t& pr, int* counter, int* status, int cg_) : cg(cg_) {
    std::memset(&p, 0, sizeof(p));
    p.a_tx_bytes = BM * BK * 2;
    p.act = device_act(pr.act);
    p.scale = pr.gate_mult * pr.down_mult;
    p.group_m = 16;
    p.counter = counter;
    p.status = status;
    p.timeout_ns = wait_limit_ns();
    p.debug_flags = g_debug_flags.load();
  }
  // K-major operand: array [rows, K] (row pitch K), box {64, box_rows}
  int kmajor(const void* ptr, int rows, int K, int box_rows) {
    if (nmaps >= MAX_MAPS) { ok = false; return 0; }
    if (!make_map(&p.maps[nmaps], ptr, K, rows, K, BK, box_rows)) ok = false;
    return nmaps++;
  }
  // K-major A operand [rows, K]: an output with fewer than 128 rows loads
  // boxes of its rows only (rounded up to 16); the MMA's rows beyond them
  // read stale shared memory and only produce accumulator rows past the
  // output, which the epilogue never stores.
  int kmajor_a(const void* ptr, int rows, int K) {
    const int box = rows < BM ? ((rows + 15) / 16) * 16 : BM;
    p.a_tx_bytes = box * BK * 2;
    return kmajor(ptr, rows, K, box);
  }
  // MN-major operand: array [K, MN] (row pitch MN), box {64, 64}
  int mnmajor(const void* ptr, int K, int MN) {
    if (nmaps >= MAX_MAPS) { ok = false; return 0; }
    if (!make_map(&p.maps[nmaps], ptr, MN, K, MN, 64, BK)) ok = false;
    return nmaps++;
  }
  // e4m3 operands [rows, K] (K bytes per row), boxes {128 k, box_rows}; the
  // A operand's boxes are row-sized below 128 rows, as in kmajor_a.
  int kmajor_u8(const void* ptr, int rows, int K, int box_rows) {
    if (nmaps >= MAX_MAPS) { ok = false; return 0; }
    if (!make_map(&p.maps[nmaps], ptr, K, rows, K, 2 * BK, box_rows, 2)) ok = false;
    return nmaps++;
  }
  int kmajor_a_u8(const void* ptr, int rows, int K) {
    const int box = rows < BM ? ((rows + 15) / 16) * 16 : BM;
    p.a_tx_bytes = box * BK * 2;  // 128 bytes per row, as for bf16
    return kmajor_u8(ptr, rows, K, box);
  }
  // 8-bit MN-major operand [K, MN] (MN bytes per row), boxes {128 mn, 128 k}
  int mnmajor_u8(const void* ptr, int K, int MN) {
    if (nmaps >= MAX_MAPS) { ok = false; return 0; }
    if (!make_map(&p.maps[nmaps], ptr, MN, K, MN, 2 * BK, 2 * BK, 2)) ok = false;
    return nmaps++;
  }
  // bf16 input [rows, cols] of a derivative epilogue, boxes {256, 128}: the
  // producer prefetches each tile's rows into L2 ahead of the epilogue
  int prefetch_map(const void* ptr, int rows, int cols) {
    if (!ptr) return -1;
    if (nmaps >= MAX_MAPS) { ok = false; return -1; }
    if (!make_map(&p.maps[nmaps], ptr, cols, rows, cols, MMA_N, BM, 0, CU_TENSOR_MAP_SWIZZLE_NONE))
      ok = false;
    return nmaps++;
  }
  // 8-bit epilogue output [rows, cols]: one 32-row x 128-byte box per warp
  // and tile, 128-byte swizzle; half = true: 32-row x 64-byte boxes, two per
  // warp and tile, 64-byte swizzle.
  int output_u8(void* ptr, int rows, int cols, bool half = false) {
    if (!ptr) return -1;
    if (nmaps >= MAX_MAPS) { ok = false; return -1; }
    if (!make_map(&p.maps[nmaps], ptr, cols, rows, cols, half ? 64 : 128, 32, 2,
                  half ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
      ok = false;
    return nmaps++;
  }
  // Epilogue output [rows, cols] (row pitch cols), stored in 32 x 32 boxes;
  // -1 when the output is not requested.
  int output(void* ptr, int rows, int cols, bool f32 = false) {
    if (!ptr) return -1;
    if (nmaps >= MAX_MAPS) { ok = false; return -1; }
    if (!make_map(&p.maps[nmaps], ptr, cols, rows, cols, 32, 32, f32,
                  f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      ok = false;
    return nmaps++;
  }
  // ke: K elements per k-block (bf16 64, e4m3 128: a 128-byte row either way)
  Prob& add(int M, int N, int K0, int K1, int tile_n, int ksplit = 1, int ke = BK) {
    Prob& P = p.prob[p.nprob++];
    P.M = M;
    P.N = N;
    P.kb0 = (K0 + ke - 1) / ke;
    P.kb1 = (K1 + ke - 1) / ke;
    P.tiles_m = (M + BM * cg - 1) / (BM * cg);
    P.tiles_n = (N + tile_n - 1) / tile_n;
    const int kbt = P.kb0 + P.kb1;
    if (ksplit < 1) ksplit = 1;
    if (ksplit > kbt) ksplit = kbt;
    P.kper = (kbt + ksplit - 1) / ksplit;
    P.ksplit = (kbt + P.kper - 1) / P.kper;  // no empty splits
    P.unit_begin = p.total_units;
    P.units = P.tiles_m * P.tiles_n * P.ksplit;
    p.total_units += P.units;
    P.ld = N;
    P.mapO[0] = P.mapO[1] = P.mapO[2] = -1;
    P.mapI0 = P.mapI1 = -1;
    P.mapE = -1;
    P.l2a = P.l2b = 0;
    return P;
  }
  // B rows per K-major box: a CTA stages 256 / cg of the 256 B rows
  int b_rows() const { return MMA_N / cg; }
};

struct Call {
  cudaStream_t stream;
  int* status;
  int* counters;
  int next_counter = 0;
  int launches = 0;
  int* counter() { return counters + (next_counter++ % MAX_COUNTERS); }
  bool pdl() { return launches++ > 0; }  // the first kernel follows the memset or the caller's work
};

int cuda_err(cudaError_t e) { return e == cudaSuccess ? MLP_OK : MLP_ERR_CUDA; }

// A second stream per device for GEMMs that may run beside the caller's
// (the weight gradients beside dx), with the events of the fork and the
// join.  `mu` is held from the fork to the join so that concurrent calls do
// not interleave their records and waits.
struct Side {
  std::mutex mu;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool ok = false;
};
Side g_side[64];
std::mutex g_side_mu;

// The current device's side stream, created on first use; nullptr when it
// cannot be had (no device, creation failed, or first asked for while
// `caller` is being captured into a graph).
Side* side_stream(cudaStream_t caller) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  Side& sd = g_side[dev];
  std::lock_guard<std::mutex> lk(g_side_mu);
  if (sd.ok) return &sd;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(caller, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return nullptr;
  if (cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
  if (cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess)
    return nullptr;
  sd.ok = true;
  return &sd;
}

// ------------------------------------------------------------ tracing
// When enabled, every kernel launch is bracketed by a pair of CUDA events on
// its stream; mlp_trace_read returns (kernel tag, milliseconds) per launch.
struct TraceRec {
  int tag;
  cudaEvent_t a, b;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::atomic<bool> g_trace_flag{false};  // g_trace_on, readable without the lock
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t trace_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

template <class F>
int traced(int tag, cudaStream_t s, F&& launch) {
  std::unique_lock<std::mutex> lk(g_trace_mu);
  if (!g_trace_on) {
    lk.unlock();
    return cuda_err(launch());
  }
  TraceRec r{tag, trace_event(), trace_event()};
  if (!r.a || !r.b) return MLP_ERR_CUDA;
  if (cudaEventRecord(r.a, s) != cudaSuccess) return MLP_ERR_CUDA;
  cudaError_t e = launch();
  if (cudaEventRecord(r.b, s) != cudaSuccess) return MLP_ERR_CUDA;
  g_trace.push_back(r);
  return cuda_err(e);
}

// Co-resident CTA groups of a kernel instance on the current device (cached).
template <int EPI, bool A_MN, bool B_MN, int CG, int ACT>
int groups_cached() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    int v = cache[dev].load();
    if (v > 0) return v;
  }
  int v = max_groups<EPI, A_MN, B_MN, CG, ACT>();
  if (v > 0 && dev >= 0 && dev < 64) cache[dev].store(v);
  return v;
}

template <int EPI, bool A_MN, bool B_MN, int ACT>
int run_act(Gemm& g, Call& c, int tag) {
  if (!g.ok) return MLP_ERR_CUDA;
  if (g.p.total_units == 0) return MLP_OK;
  g.p.nmaps = g.nmaps;
  const bool pdl = c.pdl();
  if (g.cg == 2) {
    const int groups = groups_cached<EPI, A_MN, B_MN, 2, ACT>();
    if (groups <= 0) return MLP_ERR_CUDA;
    const int n = g.p.total_units < groups ? g.p.total_units : groups;
    return traced(tag, c.stream,
                  [&] { return launch_gemm<EPI, A_MN, B_MN, 2, ACT>(g.p, 2 * n, c.stream, pdl); });
  }
  if constexpr (EPI == EPI_FWD_FUSED) {
    return MLP_ERR_UNSUPPORTED;  // CTA pairs only
  } else {
    const int sms = num_sms();
    const int n = g.p.total_units < sms ? g.p.total_units : sms;
    return traced(tag, c.stream, [&] {
      return launch_gemm<EPI, A_MN, B_MN, 1, ACT>(g.p, n < 1 ? 1 : n, c.stream, pdl);
    });
  }
}

// Kernels without an activation epilogue.
template <int EPI, bool A_MN, bool B_MN>
int run(Gemm& g, Call& c, int tag) {
  return run_act<EPI, A_MN, B_MN, 0>(g, c, tag);
}

// Activation epilogues: one kernel instance per activation.
template <int EPI, bool A_MN, bool B_MN>
int run_gated(Gemm& g, Call& c, int tag) {
  switch (g.p.act) {
    case ACT_RELU: return run_act<EPI, A_MN, B_MN, ACT_RELU>(g, c, tag);
    case ACT_GELU_TANH: return run_act<EPI, A_MN, B_MN, ACT_GELU_TANH>(g, c, tag);
    case ACT_SIGMOID: return run_act<EPI, A_MN, B_MN, ACT_SIGMOID>(g, c, tag);
    default: return run_act<EPI, A_MN, B_MN, ACT_SILU>(g, c, tag);
  }
}
template <int EPI, bool A_MN, bool B_MN>
int run_nongated(Gemm& g, Call& c, int tag) {
  switch (g.p.act) {
    case ACT_RELU: return run_act<EPI, A_MN, B_MN, ACT_RELU>(g, c, tag);
    case ACT_GELU_TANH: return run_act<EPI, A_MN, B_MN, ACT_GELU_TANH>(g, c, tag);
    default: return run_act<EPI, A_MN, B_MN, ACT_RELU_SQ>(g, c, tag);
  }
}

// ------------------------------------------------------------ validation
int check_problem(const mlp_problem_t* p) {
  if (!p) return MLP_ERR_INVALID_ARG;
  if (p->M <= 0 || p->H <= 0 || p->I <= 0) return MLP_ERR_INVALID_ARG;
  if (p->act < MLP_ACT_SWIGLU || p->act > MLP_ACT_GLU) return MLP_ERR_INVALID_ARG;
  if (!std::isfinite(p->gate_mult) || !std::isfinite(p->down_mult)) return MLP_ERR_INVALID_ARG;
  if (p->H % 8 || p->I % 8) return MLP_ERR_ALIGNMENT;
  // TMA coordinates and tile counts are 32-bit
  if ((long long)p->M * p->I >= (1LL << 40) || (long long)p->M * p->H >= (1LL << 40))
    return MLP_ERR_UNSUPPORTED;
  return MLP_OK;
}

bool gated(const mlp_problem_t* p) {
  return p->act == MLP_ACT_SWIGLU || p->act == MLP_ACT_REGLU || p->act == MLP_ACT_GEGLU ||
         p->act == MLP_ACT_GLU;
}

size_t inter_bytes(const mlp_problem_t* p) { return round256((size_t)p->M * p->I * 2); }

// Split-K factor of a bf16-output GEMM [rows, cols] x K whose output tiles
// cannot fill the GPU: the splits' fp32 partial sums meet in a zeroed region
// of the workspace (TMA reduce-add) and one elementwise pass converts it to
// bf16.  It depends on the shape only (a nominal 152 SMs), so the workspace
// size does too.
//  - Decode-sized token counts (at most 32 tiles of 128 x 256): about 128
//    work units with at least 8 k-blocks each.
//  - `fill` (the forward's down projection): when its 256 x 256 tiles (CTA
//    pairs) would occupy at most half of the 76 pairs, the smallest split
//    whose units fill at least 80 % of their last wave, again with at least
//    8 k-blocks a unit.  (A 512-token Llama-3-8B down projection is 32 such
//    tiles.)  Measured against the unsplit forward (the gated forward then
//    runs as one launch): 9-13 % faster at 384 and 512 tokens of the
//    4096-wide shapes, 3-10 % at 640-1024 tokens of a 2048-wide one; with
//    more tiles, splitting until the units filled their waves lost to the
//    one-launch forward.  The backward's dx is left whole: its last wave
//    shares the GPU with the weight gradients on the second stream.
constexpr int SPLIT_NOMINAL_SMS = 152;
int bf16_split(int rows, int cols, int K, bool fill) {
  const long long tiles =
      (long long)((rows + BM - 1) / BM) * (long long)((cols + MMA_N - 1) / MMA_N);
  const int kb = (K + BK - 1) / BK;
  if (kb < 16) return 1;
  if (tiles <= 32) {
    int split = static_cast<int>(128 / tiles);
    if (split > kb / 8) split = kb / 8;
    return split < 2 ? 1 : split;
  }
  if (!fill) return 1;
  // 256 x 256 tiles on CTA pairs (rows > 128 take pairs)
  const int pairs = SPLIT_NOMINAL_SMS / 2;
  const long long ptiles =
      (long long)((rows + 2 * BM - 1) / (2 * BM)) * (long long)((cols + MMA_N - 1) / MMA_N);
  if (2 * ptiles > pairs) return 1;
  for (int s = 2; s <= 8 && kb / s >= 8; ++s) {
    const long long units = ptiles * s;
    const long long waves = (units + pairs - 1) / pairs;
    if (units * 5 >= waves * pairs * 4) return s;
  }
  return 1;
}

// K of the bf16-output GEMM of a mode: the down projection (forward) or dx.
int split_k_of(const mlp_problem_t* p, int mode) {
  if (mode == MLP_MODE_FWD || mode == MLP_MODE_INFER) return p->I;
  return gated(p) ? 2 * p->I : p->I;
}

// The split-K factor of a mode's [M,H] output GEMM.
int out_split_of(const mlp_problem_t* p, int mode) {
  const bool fwd = mode == MLP_MODE_FWD || mode == MLP_MODE_INFER;
  return bf16_split(p->M, p->H, split_k_of(p, mode), fwd);
}

size_t split_bytes(const mlp_problem_t* p, int mode) {
  return out_split_of(p, mode) > 1 ? round256((size_t)p->M * p->H * 4) : 0;
}

size_t ws_size(const mlp_problem_t* p, int mode) {
  // e4m3 forward: the control block + the e4m3 postact (one byte per element)
  if (mode == MLP_MODE_FP8_FWD) return CTRL_BYTES + round256((size_t)p->M * p->I);
  // 8-bit backward: + the e5m2 codes of dout [M,H] and of dpre [M,I]
  if (mode == MLP_MODE_FP8_BWD)
    return CTRL_BYTES + round256((size_t)p->M * p->H) + round256((size_t)p->M * p->I);
  size_t n = CTRL_BYTES + inter_bytes(p);  // control block + postact a
  if (mode == MLP_MODE_BWD_RECOMPUTE) n += inter_bytes(p) * (gated(p) ? 2 : 1);
  return n + split_bytes(p, mode);  // + the fp32 partial-sum region (small M only)
}

// Offset of the fp32 partial-sum region in the workspace.
size_t split_offset(const mlp_problem_t* p, int mode) { return ws_size(p, mode) - split_bytes(p, mode); }

// Required pointer present and 16-byte aligned; optional pointer aligned if present.
int need(const void* ptr) {
  if (!ptr) return MLP_ERR_INVALID_ARG;
  return aligned16(ptr) ? MLP_OK : MLP_ERR_ALIGNMENT;
}
int opt(const void* ptr) { return (!ptr || aligned16(ptr)) ? MLP_OK : MLP_ERR_ALIGNMENT; }

#define MLP_TRY(...)                 \
  do {                               \
    int _rc = (__VA_ARGS__);         \
    if (_rc != MLP_OK) return _rc;   \
  } while (0)

int check_weights(const mlp_problem_t* p, const void* Wg, const void* Wu, const void* Wd) {
  MLP_TRY(need(Wg));
  MLP_TRY(need(Wd));
  if (gated(p)) {
    MLP_TRY(need(Wu));
  } else if (Wu) {
    return MLP_ERR_INVALID_ARG;  // non-gated activations take one fc1 weight
  }
  return MLP_OK;
}

int check_block(const mlp_block_t* b) {
  if (!b) return MLP_ERR_INVALID_ARG;
  if (!std::isfinite(b->resid_lambda) || !std::isfinite(b->post_lambda) ||
      !std::isfinite(b->eps) || b->eps < 0.f)
    return MLP_ERR_INVALID_ARG;
  return MLP_OK;
}

int check_ws(const mlp_problem_t* p, int mode, const void* ws, size_t ws_bytes) {
  if (!ws) return MLP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MLP_ERR_ALIGNMENT;
  if (ws_bytes < ws_size(p, mode)) return MLP_ERR_WORKSPACE_TOO_SMALL;
  return MLP_OK;
}

// Output tiles (256 columns, 128 x cg rows) of a GEMM output [rows, cols].
long long out_tiles(int rows, int cols, int cg) {
  return (long long)((rows + BM * cg - 1) / (BM * cg)) * ((cols + MMA_N - 1) / MMA_N);
}

// Split-K factor of the weight-gradient launch: when its output tiles cannot
// fill the GPU, the token reduction (K = M) is split so that the work units
// do, with at least 8 k-blocks per unit (fp32 accumulation only: the
// partial sums meet through atomic adds in dW).
int wgrad_split(int M, long long tiles, int cg, int fuse) {
  if (!fuse || tiles <= 0) return 1;
  const int slots = num_sms() / cg;
  const int kb = (M + BK - 1) / BK;
  int ksplit = 1;
  if (tiles < slots) {
    ksplit = (int)(slots / tiles);
    while (ksplit > 1 && kb / ksplit < 8) --ksplit;
  }
  return ksplit;
}

// clear = false: the call's first kernel clears the status word itself (the
// decode weight streams, which use no counter of the control block), so the
// call enqueues no memset.
int begin_call(Call& c, void* ws, void* stream, bool clear = true) {
  c.stream = static_cast<cudaStream_t>(stream);
  c.status = static_cast<int*>(ws);
  c.counters = static_cast<int*>(ws) + COUNTER_BASE;
  return clear ? cuda_err(cudaMemsetAsync(ws, 0, CTRL_BYTES, c.stream)) : MLP_OK;
}

// The MLP block's neighbours (mlp_block_fwd / mlp_block_bwd); nullptr for
// the plain MLP.
struct Block {
  float alpha;        // the residual stream's scale (resid_lambda)
  float eps;          // the RMS norm's epsilon
  float* rstd_out;    // forward: where the per-token scale 1/r goes
  const float* rstd;  // the per-token scale the GEMM epilogues apply
};



// gate/up (or fc1) GEMM with the activation epilogue.
//   a_out: postact (may be null), G_out/U_out: preact stores (may be null)
//   rstd: per-row scale of the accumulators (the block's RMS norm; may be null)
int launch_fwd_act(const mlp_problem_t* p, Call& c, const void* x, const void* Wg, const void* Wu,
                   void* a_out, void* G_out, void* U_out, const float* rstd = nullptr) {
  Gemm g(*p, c.counter(), c.status, pick_cg(p->M));
  const int mA = g.kmajor_a(x, p->M, p->H);
  if (gated(p)) {
    const int mG = g.kmajor(Wg, p->I, p->H, 128);
    const int mU = g.kmajor(Wu, p->I, p->H, 128);
    const int oA = g.output(a_out, p->M, p->I);
    const int oG = g.output(G_out, p->M, p->I);
    const int oU = g.output(U_out, p->M, p->I);
    Prob& P = g.add(p->M, p->I, p->H, 0, 128);
    P.l2a = L2_EVICT_LAST;   // x: every tile column re-reads it
    P.l2b = L2_EVICT_FIRST;  // the weights: a panel's reuse is by consecutive row tiles
    P.mapA0 = mA;
    P.mapB0 = mG;
    P.mapB1 = mU;
    P.mapO[0] = oA;
    P.mapO[1] = oG;
    P.mapO[2] = oU;
    P.rstd = rstd;
    return run_gated<EPI_GATED_FWD, false, false>(g, c, MLP_KERNEL_GATE_UP);
  }
  const int mW = g.kmajor(Wg, p->I, p->H, g.b_rows());
  const int oA = g.output(a_out, p->M, p->I);
  const int oP = g.output(G_out, p->M, p->I);
  Prob& P = g.add(p->M, p->I, p->H, 0, MMA_N);
  P.l2b = L2_EVICT_LAST;  // W1: walked again by every group of row tiles
  P.mapA0 = mA;
  P.mapB0 = mW;
  P.mapO[0] = oA;
  P.mapO[1] = oP;
  P.rstd = rstd;
  return run_nongated<EPI_ACT_FWD, false, false>(g, c, MLP_KERNEL_GATE_UP);
}

// Non-gated recompute, stages 0 + 1 fused: per output tile, segment 0
// accumulates p = x W1^T (K = H) and segment 1 dh = dout Wd (K = H) into the
// other accumulator; the epilogue writes a = s*act(p) (if a_out) and
// dP = s*dh*act'(p).
int launch_dact_recomp(const mlp_problem_t* p, Call& c, const void* x, const void* W1,
                       const void* dout, const void* Wd, void* dP, void* a_out) {
  Gemm g(*p, c.counter(), c.status, pick_cg(p->M));
  const int mA0 = g.kmajor_a(x, p->M, p->H);
  const int mB0 = g.kmajor(W1, p->I, p->H, g.b_rows());
  const int mA1 = g.kmajor_a(dout, p->M, p->H);
  const int mB1 = g.mnmajor(Wd, p->H, p->I);  // Wd [H,I]: B(n=i, k=h) is N-contiguous
  const int oP = g.output(dP, p->M, p->I);
  const int oA = g.output(a_out, p->M, p->I);
  Prob& P = g.add(p->M, p->I, p->H, p->H, MMA_N);
  P.l2b = L2_EVICT_LAST;  // W1 and Wd: walked again by every group of row tiles
  P.mapA0 = mA0;
  P.mapB0 = mB0;
  P.mapA1 = mA1;
  P.mapB1 = mB1;
  P.mapO[0] = oP;
  P.mapO[1] = oA;
  return run_nongated<EPI_DACT_RECOMP, false, false>(g, c, MLP_KERNEL_DACT_RECOMPUTE);
}

// fp32 [n] -> bf16 [n] (the split-K partial-sum region to the output), plus
// alpha * resid when the block's residual is given.
int convert_out(Call& c, const float* part, void* out, long long n, const void* resid = nullptr,
                float alpha = 0.f) {
  const bool pdl = c.pdl();
  return traced(MLP_KERNEL_CONVERT, c.stream,
                [&] { return launch_f32_to_bf16(part, out, n, c.stream, pdl, resid, alpha); });
}

// out = a Wd^T (+ alpha * resid for the block); with split > 1 through the
// zeroed fp32 region `part`.
int launch_down(const mlp_problem_t* p, Call& c, const void* a, const void* Wd, void* out,
                float* part, int split, const void* resid = nullptr, float alpha = 0.f) {
  Gemm g(*p, c.counter(), c.status, pick_cg(p->M));
  const int mA = g.kmajor_a(a, p->M, p->I);
  const int mB = g.kmajor(Wd, p->H, p->I, g.b_rows());
  if (split > 1) {
    const int oP = g.output(part, p->M, p->H, true);
    Prob& P = g.add(p->M, p->H, p->I, 0, MMA_N, split);
    P.l2a = L2_EVICT_LAST;   // the postact: re-read by every tile column
    P.l2b = L2_EVICT_FIRST;  // Wd
    P.mapA0 = mA;
    P.mapB0 = mB;
    P.mapO[0] = oP;
    MLP_TRY(run<EPI_ACCUM_F32, false, false>(g, c, MLP_KERNEL_DOWN));
    return convert_out(c, part, out, (long long)p->M * p->H, resid, alpha);
  }
  const int oO = g.output(out, p->M, p->H);
  Prob& P = g.add(p->M, p->H, p->I, 0, MMA_N);
  P.l2a = L2_EVICT_LAST;   // the postact: re-read by every tile column
  P.l2b = L2_EVICT_FIRST;  // Wd
  P.mapA0 = mA;
  P.mapB0 = mB;
  P.mapO[0] = oO;
  P.in0 = resid;  // the epilogue reads the residual tile before storing over it
  P.alpha = alpha;
  return run<EPI_STORE_BF16, false, false>(g, c, MLP_KERNEL_DOWN);
}

// The gated forward as one launch (EPI_FWD_FUSED) on CTA pairs: problem 0
// is the gate/up GEMM (a, and G/U when saved), problem 1 the down
// projection out = a Wd^T (+ alpha * resid for the block).  A down unit
// waits until its 256-row block of a is stored; the down units are rastered
// block by block, so the first ones claimed belong to the blocks whose
// gate/up tiles finish first.  The per-block counts live in the control
// block (zeroed by begin_call).
bool fused_forward(const mlp_problem_t* p, int split) {
  return gated(p) && split == 1 && g_tile_policy.load() == 0 && pick_cg(p->M) == 2 &&
         (p->M + 2 * BM - 1) / (2 * BM) <= MAX_DEP_BLOCKS;
}

int launch_fwd_fused(const mlp_problem_t* p, Call& c, const void* x, const void* Wg,
                     const void* Wu, const void* Wd, void* a, void* G_out, void* U_out, void* out,
                     const float* rstd, const void* resid, float alpha) {
  Gemm g(*p, c.counter(), c.status, 2);
  const int mX = g.kmajor_a(x, p->M, p->H);
  const int mG = g.kmajor(Wg, p->I, p->H, 128);
  const int mU = g.kmajor(Wu, p->I, p->H, 128);
  const int oA = g.output(a, p->M, p->I);
  const int oG = g.output(G_out, p->M, p->I);
  const int oU = g.output(U_out, p->M, p->I);
  const int mA = g.kmajor_a(a, p->M, p->I);
  const int mD = g.kmajor(Wd, p->H, p->I, g.b_rows());
  const int oO = g.output(out, p->M, p->H);
  Prob& P0 = g.add(p->M, p->I, p->H, 0, 128);
  P0.l2b = L2_EVICT_LAST;  // Wg, Wu: walked again by every group of 16 row tiles
  P0.mapA0 = mX;
  P0.mapB0 = mG;
  P0.mapB1 = mU;
  P0.mapO[0] = oA;
  P0.mapO[1] = oG;
  P0.mapO[2] = oU;
  P0.rstd = rstd;
  Prob& P1 = g.add(p->M, p->H, p->I, 0, MMA_N);
  P1.mapA0 = mA;
  P1.mapB0 = mD;
  P1.mapO[0] = oO;
  P1.in0 = resid;  // the epilogue reads the residual tile before storing over it
  P1.alpha = alpha;
  P1.group_m = 1;
  g.p.dep = c.status + DEP_BASE;
  g.p.dep_target = P0.tiles_n * 2 * NUM_EPI_WARPS;  // every epilogue warp of the pair, per tile
  return run_gated<EPI_FWD_FUSED, false, false>(g, c, MLP_KERNEL_FWD_FUSED);
}

int forward(const mlp_problem_t* p, const void* x, const void* Wg, const void* Wu, const void* Wd,
            void* out, void* G_save, void* U_save, void* ws, size_t ws_bytes, void* stream,
            int mode, const Block* blk = nullptr) {
  MLP_TRY(check_problem(p));
  MLP_TRY(need(x));
  MLP_TRY(check_weights(p, Wg, Wu, Wd));
  MLP_TRY(need(out));
  MLP_TRY(opt(G_save));
  MLP_TRY(opt(U_save));
  if (!gated(p) && U_save) return MLP_ERR_INVALID_ARG;
  MLP_TRY(check_ws(p, mode, ws, ws_bytes));
  const int dk = blk ? 0 : decode_kernel(p);
  Call c;
  MLP_TRY(begin_call(c, ws, stream, dk == 0));
  void* a = static_cast<char*>(ws) + CTRL_BYTES;
  if (dk != 0) {
    // a few tokens: two weight-streaming passes (warp-level MMA, or CUDA
    // cores); the first, launched after everything before it on the stream,
    // clears the status word in place of the control block's memset
    const bool pdl0 = c.pdl();
    MLP_TRY(traced(MLP_KERNEL_GATE_UP, c.stream, [&] {
      return dk == 2 ? launch_decode_mma_act(x, Wg, Wu, a, G_save, U_save, p->M, p->H, p->I,
                                             device_act(p->act), gated(p),
                                             p->gate_mult * p->down_mult, c.stream, pdl0, c.status)
                     : launch_decode_act(x, Wg, Wu, a, G_save, U_save, p->M, p->H, p->I,
                                         device_act(p->act), gated(p),
                                         p->gate_mult * p->down_mult, c.stream, pdl0, c.status);
    }));
    const bool pdl1 = c.pdl();
    return traced(MLP_KERNEL_DOWN, c.stream, [&] {
      return dk == 2 ? launch_decode_mma_down(a, Wd, out, p->M, p->H, p->I, c.stream, pdl1)
                     : launch_decode_down(a, Wd, out, p->M, p->H, p->I, c.stream, pdl1);
    });
  }
  const int split = out_split_of(p, mode);
  float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + split_offset(p, mode));
  if (split > 1)
    MLP_TRY(cuda_err(cudaMemsetAsync(part, 0, (size_t)p->M * p->H * 4, c.stream)));
  if (blk) {
    // the block's RMS norm: 1/r per token, applied in the gate/up epilogue
    const bool pdl = c.pdl();
    MLP_TRY(traced(MLP_KERNEL_RSTD, c.stream, [&] {
      return launch_rstd(x, blk->rstd_out, p->M, p->H, blk->eps, c.stream, pdl);
    }));
  }
  if (fused_forward(p, split))
    return launch_fwd_fused(p, c, x, Wg, Wu, Wd, a, G_save, U_save, out,
                            blk ? blk->rstd : nullptr, blk ? x : nullptr, blk ? blk->alpha : 0.f);
  MLP_TRY(launch_fwd_act(p, c, x, Wg, Wu, a, G_save, U_save, blk ? blk->rstd : nullptr));
  return launch_down(p, c, a, Wd, out, part, split, blk ? x : nullptr, blk ? blk->alpha : 0.f);
}

int backward(const mlp_problem_t* p, const void* dout, const void* x, const void* Wg,
             const void* Wu, const void* Wd, void* G, void* U, void* dx, void* dWg, void* dWu,
             void* dWd, int fuse, void* ws, size_t ws_bytes, void* stream, bool recompute,
             const Block* blk = nullptr) {
  MLP_TRY(check_problem(p));
  if (fuse != 0 && fuse != 1) return MLP_ERR_INVALID_ARG;
  MLP_TRY(need(dout));
  MLP_TRY(need(x));
  MLP_TRY(check_weights(p, Wg, Wu, Wd));
  if (!recompute) {
    MLP_TRY(need(G));
    if (gated(p)) {
      MLP_TRY(need(U));
    } else if (U) {
      return MLP_ERR_INVALID_ARG;
    }
  }
  MLP_TRY(opt(dx));
  MLP_TRY(opt(dWg));
  MLP_TRY(opt(dWu));
  MLP_TRY(opt(dWd));
  if (!gated(p) && dWu) return MLP_ERR_INVALID_ARG;
  const int mode = recompute ? MLP_MODE_BWD_RECOMPUTE : MLP_MODE_BWD;
  MLP_TRY(check_ws(p, mode, ws, ws_bytes));

  const bool need_dact = dx || dWg || dWu;
  if (!need_dact && !dWd) return MLP_OK;  // nothing requested

  Call c;
  MLP_TRY(begin_call(c, ws, stream));
  char* base = static_cast<char*>(ws) + CTRL_BYTES;
  const int dx_split = dx ? out_split_of(p, mode) : 1;
  float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + split_offset(p, mode));
  if (dx_split > 1)
    MLP_TRY(cuda_err(cudaMemsetAsync(part, 0, (size_t)p->M * p->H * 4, c.stream)));
  void* a = base;  // postact (input of dWd)
  // non-gated recompute: the preact and its derivative in one kernel
  const bool fused_recomp = recompute && !gated(p) && need_dact;
  if (recompute) {
    G = base + inter_bytes(p);
    U = gated(p) ? base + 2 * inter_bytes(p) : nullptr;
    // stage 0: recompute the preacts (quack MLPRecomputeFunc: preact = x W1^T);
    // the postact needed by dWd comes straight from the fp32 accumulators
    if (fused_recomp) {
      MLP_TRY(launch_dact_recomp(p, c, x, Wg, dout, Wd, G, dWd ? a : nullptr));
    } else {
      MLP_TRY(launch_fwd_act(p, c, x, Wg, Wu, dWd ? a : nullptr, G, U));
    }
  }
  const int M = p->M, H = p->H, I = p->I;

  if (need_dact && !fused_recomp) {
    // stage 1: dh = dout Wd (K = H); epilogue writes dG, dU over G, U (and the
    // postact a when the saved preacts are the only source of it)
    Gemm g(*p, c.counter(), c.status, pick_cg(M));
    const int mA = g.kmajor_a(dout, M, H);
    const int mB = g.mnmajor(Wd, H, I);  // Wd [H,I]: B(n=i, k=h) is N-contiguous
    void* a_out = (dWd && !recompute) ? a : nullptr;
    const int oG = g.output(G, M, I);
    const int oU = gated(p) ? g.output(U, M, I) : -1;
    const int oA = g.output(a_out, M, I);
    // (no L2 prefetch of G/U here: with the long K of these GEMMs the
    // epilogue keeps up, and the prefetch made the kernel 5-7 % slower)
    Prob& P = g.add(M, I, H, 0, MMA_N);
    P.l2a = L2_EVICT_LAST;  // dout: re-read by every tile column
    P.mapA0 = mA;
    P.mapB0 = mB;
    P.in0 = G;
    P.in1 = U;
    P.rstd = blk ? blk->rstd : nullptr;  // dG, dU (dP) come out times 1/r
    // gated: dG, dU, a;  non-gated: dP, a
    P.mapO[0] = oG;
    if (gated(p)) {
      P.mapO[1] = oU;
      P.mapO[2] = oA;
    } else {
      P.mapO[1] = oA;
    }
    MLP_TRY(gated(p) ? run_gated<EPI_DGATED, false, true>(g, c, MLP_KERNEL_DGATED)
                     : run_nongated<EPI_DACT, false, true>(g, c, MLP_KERNEL_DGATED));
  } else if (!recompute) {
    // only dWd requested: rebuild the postact without the derivative
    const bool pdl = c.pdl();
    MLP_TRY(traced(MLP_KERNEL_POSTACT, c.stream, [&] {
      return launch_postact(G, U, a, (long long)M * I, device_act(p->act),
                            p->gate_mult * p->down_mult, c.stream, pdl);
    }));
  }
  void* dG = G;
  void* dU = U;

  // Stages 2 and 3 read only what stage 1 wrote (and the inputs).  With both
  // requested, the weight gradients go to the side stream, forked after
  // stage 1 and joined before the call returns: dx, enqueued first and
  // launched early through PDL, takes the SMs, and the weight-gradient CTAs
  // take those that dx's last, partial wave of tiles leaves idle.
  // (With tracing on, kernels run one after another so that each traced
  // duration is the kernel's own.)
  const bool want_w = dWg || dWu || dWd;
  Side* side = (dx && want_w && !g_trace_flag.load()) ? side_stream(c.stream) : nullptr;
  std::unique_lock<std::mutex> side_lk;
  if (side) {
    side_lk = std::unique_lock<std::mutex>(side->mu);
    MLP_TRY(cuda_err(cudaEventRecord(side->fork, c.stream)));
  }

  if (dx) {
    // stage 2: dx = [dG|dU] [Wg;Wu], one accumulator over K = 2I (non-gated: K = I)
    Gemm g(*p, c.counter(), c.status, pick_cg(M));
    const int mA0 = g.kmajor_a(dG, M, I);
    const int mB0 = g.mnmajor(Wg, I, H);  // Wg [I,H]: B(n=h, k=i) is N-contiguous
    int mA1 = 0, mB1 = 0;
    if (gated(p)) {
      mA1 = g.kmajor_a(dU, M, I);
      mB1 = g.mnmajor(Wu, I, H);
    }
    const int oX = dx_split > 1 ? g.output(part, M, H, true) : g.output(dx, M, H);
    Prob& P = g.add(M, H, I, gated(p) ? I : 0, MMA_N, dx_split);
    P.l2a = L2_EVICT_LAST;   // dG, dU: re-read by every tile column
    P.l2b = L2_EVICT_FIRST;  // Wg, Wu
    P.mapA0 = mA0;
    P.mapB0 = mB0;
    P.mapA1 = mA1;
    P.mapB1 = mB1;
    P.mapO[0] = oX;
    if (dx_split > 1) {
      MLP_TRY((run<EPI_ACCUM_F32, false, true>(g, c, MLP_KERNEL_DX)));
      MLP_TRY(convert_out(c, part, dx, (long long)M * H));
    } else {
      MLP_TRY((run<EPI_STORE_BF16, false, true>(g, c, MLP_KERNEL_DX)));
    }
    if (blk) {
      // the block: dx holds D = dn / r; through the RMS norm and the residual
      const bool pdl = c.pdl();
      MLP_TRY(traced(MLP_KERNEL_RMSNORM_BWD, c.stream, [&] {
        return launch_rmsnorm_bwd(dx, x, dout, blk->rstd, M, H, blk->alpha, c.stream, pdl);
      }));
    }
  }

  if (want_w) {
    // stage 3: weight gradients in one grouped launch, reduced over the M tokens:
    //   dWg = dG^T x, dWu = dU^T x  ([I,H])   dWd = dout^T a  ([H,I])
    Call cw = c;  // same control block; the side stream when forked
    if (side) {
      cw.stream = side->stream;
      cw.launches = 0;  // its first kernel follows an event wait, not a kernel
      MLP_TRY(cuda_err(cudaStreamWaitEvent(side->stream, side->fork, 0)));
    }
    Gemm g(*p, c.counter(), c.status, pick_cg(H < I ? H : I));
    struct W { const void* A; int rows; const void* B; int cols; void* out; };
    W list[3];
    int n = 0;
    if (dWg) list[n++] = {dG, I, x, H, dWg};
    if (dWu) list[n++] = {dU, I, x, H, dWu};
    if (dWd) list[n++] = {dout, H, a, I, dWd};
    long long tiles = 0;
    for (int i = 0; i < n; ++i) tiles += out_tiles(list[i].rows, list[i].cols, g.cg);
    const int ksplit = wgrad_split(M, tiles, g.cg, fuse);
    for (int i = 0; i < n; ++i) {
      const int mA = g.mnmajor(list[i].A, M, list[i].rows);
      const int mB = g.mnmajor(list[i].B, M, list[i].cols);
      const int oW = g.output(list[i].out, list[i].rows, list[i].cols, fuse != 0);
      Prob& P = g.add(list[i].rows, list[i].cols, M, 0, MMA_N, ksplit);
      P.l2b = L2_EVICT_LAST;  // x, or the postact: shared by the three problems' tile rows
      P.mapA0 = mA;
      P.mapB0 = mB;
      P.mapO[0] = oW;
    }
    if (fuse) {
      MLP_TRY((run<EPI_ACCUM_F32, true, true>(g, cw, MLP_KERNEL_WGRAD)));
    } else {
      MLP_TRY((run<EPI_STORE_BF16, true, true>(g, cw, MLP_KERNEL_WGRAD)));
    }
    if (side) {
      MLP_TRY(cuda_err(cudaEventRecord(side->join, side->stream)));
      MLP_TRY(cuda_err(cudaStreamWaitEvent(c.stream, side->join, 0)));
    }
  }
  return MLP_OK;
}

}  // namespace

extern "C" {

size_t mlp_workspace_size(const mlp_problem_t* p, int mode) {
  if (check_problem(p) != MLP_OK) return 0;
  if (mode < MLP_MODE_FWD || mode > MLP_MODE_FP8_BWD) return 0;
  return ws_size(p, mode);
}

int mlp_fwd(const mlp_problem_t* p, const void* x, const void* Wg, const void* Wu, const void* Wd,
            void* out, void* G_save, void* U_save, void* ws, size_t ws_bytes, void* stream) {
  return forward(p, x, Wg, Wu, Wd, out, G_save, U_save, ws, ws_bytes, stream, MLP_MODE_FWD);
}

int mlp_fwd_infer(const mlp_problem_t* p, const void* x, const void* Wg, const void* Wu,
                  const void* Wd, void* out, void* ws, size_t ws_bytes, void* stream) {
  return forward(p, x, Wg, Wu, Wd, out, nullptr, nullptr, ws, ws_bytes, stream, MLP_MODE_INFER);
}

int mlp_block_fwd(const mlp_problem_t* p, const mlp_block_t* b, const void* x, const void* Wg,
                  const void* Wu, const void* Wd, void* y, void* G_save, void* U_save,
                  float* rstd_save, void* ws, size_t ws_bytes, void* stream) {
  MLP_TRY(check_problem(p));
  MLP_TRY(check_block(b));
  MLP_TRY(need(rstd_save));
  mlp_problem_t q = *p;
  q.down_mult *= b->post_lambda;  // post_lambda scales the MLP output
  const Block blk{b->resid_lambda, b->eps, rstd_save, rstd_save};
  return forward(&q, x, Wg, Wu, Wd, y, G_save, U_save, ws, ws_bytes, stream, MLP_MODE_FWD, &blk);
}

int mlp_block_bwd(const mlp_problem_t* p, const mlp_block_t* b, const void* dy, const void* x,
                  const void* Wg, const void* Wu, const void* Wd, void* G, void* U,
                  const float* rstd, void* dx, void* dWg, void* dWu, void* dWd,
                  int fuse_grad_accum, void* ws, size_t ws_bytes, void* stream) {
  MLP_TRY(check_problem(p));
  MLP_TRY(check_block(b));
  MLP_TRY(need(rstd));
  // dx is written while the weight gradients (on the second stream) and
  // the RMS-norm pass still read x and dy
  if (dx && (dx == x || dx == dy)) return MLP_ERR_INVALID_ARG;
  mlp_problem_t q = *p;
  q.down_mult *= b->post_lambda;
  const Block blk{b->resid_lambda, b->eps, nullptr, rstd};
  return backward(&q, dy, x, Wg, Wu, Wd, G, U, dx, dWg, dWu, dWd, fuse_grad_accum, ws, ws_bytes,
                  stream, false, &blk);
}

int mlp_fp8_quantize(const void* src, long long n, const float* scale, void* dst, float* amax,
                     void* stream) {
  if (n < 0 || (n % 8) != 0) return MLP_ERR_INVALID_ARG;
  if (n == 0) return MLP_OK;
  MLP_TRY(need(src));
  MLP_TRY(need(dst));
  if (!scale) return MLP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return traced(MLP_KERNEL_QUANT, s,
                [&] { return launch_quant_f8(src, n, scale, dst, amax, F8_E4M3, s, false); });
}

int mlp_fp8_fwd(const mlp_problem_t* p, const void* x8, const void* W1_8, const void* W2_8,
                const float* scales, void* out, void* a8_save, void* pre_save, float* amax_a,
                void* ws, size_t ws_bytes, void* stream) {
  MLP_TRY(check_problem(p));
  if (p->act != MLP_ACT_RELU_SQ) return MLP_ERR_UNSUPPORTED;
  if (p->H % 16 || p->I % 16) return MLP_ERR_ALIGNMENT;  // 16-byte e4m3 rows
  MLP_TRY(need(x8));
  MLP_TRY(need(W1_8));
  MLP_TRY(need(W2_8));
  MLP_TRY(need(out));
  MLP_TRY(opt(a8_save));
  MLP_TRY(opt(pre_save));
  if (!scales) return MLP_ERR_INVALID_ARG;
  MLP_TRY(check_ws(p, MLP_MODE_FP8_FWD, ws, ws_bytes));
  Call c;
  MLP_TRY(begin_call(c, ws, stream));
  void* a8 = a8_save ? a8_save : static_cast<char*>(ws) + CTRL_BYTES;
  const int M = p->M, H = p->H, I = p->I;
  {
    // fc1 on e4m3 codes, ReLU^2, the postact re-quantised with s_post
    Gemm g(*p, c.counter(), c.status, pick_cg(M));
    const int mA = g.kmajor_a_u8(x8, M, H);
    const int mB = g.kmajor_u8(W1_8, I, H, g.b_rows());
    const int oA = g.output_u8(a8, M, I, true);  // the fc1 epilogue stores half tiles
    const int oP = g.output(pre_save, M, I);
    Prob& P = g.add(M, I, H, 0, MMA_N, 1, 2 * BK);
    P.mapA0 = mA;
    P.mapB0 = mB;
    P.mapO[0] = oA;
    P.mapO[1] = oP;
    P.sa = scales + 0;  // sx
    P.sb = scales + 1;  // s1
    P.sq = scales + 3;  // s_post
    P.mult = p->gate_mult;
    P.amax = amax_a;
    MLP_TRY((run_act<EPI_ACT_FWD_F8, false, false, ACT_RELU_SQ>(g, c, MLP_KERNEL_GATE_UP)));
  }
  // the down projection on the re-quantised postact, dequantised to bf16
  Gemm g(*p, c.counter(), c.status, pick_cg(M));
  const int mA = g.kmajor_a_u8(a8, M, I);
  const int mB = g.kmajor_u8(W2_8, H, I, g.b_rows());
  const int oO = g.output(out, M, H);
  Prob& P = g.add(M, H, I, 0, MMA_N, 1, 2 * BK);
  P.mapA0 = mA;
  P.mapB0 = mB;
  P.mapO[0] = oO;
  P.sa = scales + 3;  // s_post
  P.sb = scales + 2;  // s2
  P.mult = p->down_mult;
  return run<EPI_STORE_BF16_F8, false, false>(g, c, MLP_KERNEL_DOWN);
}

int mlp_fp8_bwd(const mlp_problem_t* p, const void* dout, const void* x8, const void* W1_8,
                const void* W2_8, const void* pre, const void* a8, const float* scales, void* dx,
                void* dW1, void* dW2, float* amax_dpre, void* ws, size_t ws_bytes, void* stream) {
  MLP_TRY(check_problem(p));
  if (p->act != MLP_ACT_RELU_SQ) return MLP_ERR_UNSUPPORTED;
  if (p->H % 16 || p->I % 16) return MLP_ERR_ALIGNMENT;
  MLP_TRY(need(dout));
  MLP_TRY(opt(dx));
  MLP_TRY(opt(dW1));
  MLP_TRY(opt(dW2));
  if (!scales) return MLP_ERR_INVALID_ARG;
  const bool need_dpre = dx || dW1;
  if (need_dpre) {
    MLP_TRY(need(W2_8));
    MLP_TRY(opt(pre));
    if (!pre) {  // the derivative GEMM recomputes the preact from the forward's operands
      MLP_TRY(need(x8));
      MLP_TRY(need(W1_8));
    }
  }
  if (dx) MLP_TRY(need(W1_8));
  if (dW1) MLP_TRY(need(x8));
  if (dW2) MLP_TRY(need(a8));
  MLP_TRY(check_ws(p, MLP_MODE_FP8_BWD, ws, ws_bytes));
  if (!need_dpre && !dW2) return MLP_OK;  // nothing requested
  const int M = p->M, H = p->H, I = p->I;
  Call c;
  MLP_TRY(begin_call(c, ws, stream));
  char* base = static_cast<char*>(ws) + CTRL_BYTES;
  void* dout8 = base;
  void* dP8 = base + round256((size_t)M * H);
  // the 8-bit operands: A the e5m2 gradient codes, B the e4m3 weight / activation codes
  const int fmts = F8_E5M2 | (F8_E4M3 << 3);
  {
    // dout -> e5m2 with the static gradient scale sg
    const bool pdl = c.pdl();
    MLP_TRY(traced(MLP_KERNEL_QUANT, c.stream, [&] {
      return launch_quant_f8(dout, (long long)M * H, scales + 4, dout8, nullptr, F8_E5M2, c.stream,
                             pdl);
    }));
  }
  if (need_dpre && !pre) {
    // the same derivative with the preact recomputed in each output tile:
    // segment 0 accumulates x8 W1_8^T (both e4m3, B K-major), segment 1
    // dout8 W2_8 (e5m2 x e4m3, B MN-major); dpre = gate_mult * down_mult * sg
    // * s2 * acc1 * 2 relu(sx * s1 * acc0), to e5m2 with s_dpre
    Gemm g(*p, c.counter(), c.status, pick_cg(M));
    g.p.f8_formats = fmts;
    g.p.f8_formats0 = F8_E4M3 | (F8_E4M3 << 3);
    const int mA0 = g.kmajor_a_u8(x8, M, H);
    const int mB0 = g.kmajor_u8(W1_8, I, H, g.b_rows());
    const int mA1 = g.kmajor_a_u8(dout8, M, H);
    const int mB1 = g.mnmajor_u8(W2_8, H, I);
    const int oP = g.output_u8(dP8, M, I);
    Prob& P = g.add(M, I, H, H, MMA_N, 1, 2 * BK);
    P.mapA0 = mA0;
    P.mapB0 = mB0;
    P.mapA1 = mA1;
    P.mapB1 = mB1;
    P.mapO[0] = oP;
    P.sa = scales + 4;   // sg
    P.sb = scales + 2;   // s2
    P.sq = scales + 5;   // s_dpre
    P.sp0 = scales + 0;  // sx
    P.sp1 = scales + 1;  // s1
    P.mult = p->gate_mult * p->down_mult;
    P.amax = amax_dpre;
    MLP_TRY((run<EPI_DGRAD_F8_RECOMP, false, false>(g, c, MLP_KERNEL_DGATED)));
  } else if (need_dpre) {
    // dpre = gate_mult * down_mult * sg * s2 * (dout8 W2_8) * 2 relu(pre), to
    // e5m2 with the delayed scale s_dpre; W2_8 [H,I]: B(n=i, k=h) is N-contiguous
    Gemm g(*p, c.counter(), c.status, pick_cg(M));
    g.p.f8_formats = fmts;
    const int mA = g.kmajor_a_u8(dout8, M, H);
    const int mB = g.mnmajor_u8(W2_8, H, I);
    const int oP = g.output_u8(dP8, M, I);
    const int iP = g.prefetch_map(pre, M, I);
    const int eP = g.output(const_cast<void*>(pre), M, I);  // the epilogue's preact boxes
    Prob& P = g.add(M, I, H, 0, MMA_N, 1, 2 * BK);
    P.mapA0 = mA;
    P.mapB0 = mB;
    P.mapO[0] = oP;
    P.in0 = pre;
    P.mapI0 = iP;
    P.mapE = eP;
    P.sa = scales + 4;  // sg
    P.sb = scales + 2;  // s2
    P.sq = scales + 5;  // s_dpre
    P.mult = p->gate_mult * p->down_mult;
    P.amax = amax_dpre;
    MLP_TRY((run<EPI_DGRAD_F8, false, true>(g, c, MLP_KERNEL_DGATED)));
  }
  // dx and the weight gradients read only the codes above and the inputs:
  // with both requested, the weight gradients run on the side stream
  const bool want_w = dW1 || dW2;
  Side* side = (dx && want_w && !g_trace_flag.load()) ? side_stream(c.stream) : nullptr;
  std::unique_lock<std::mutex> side_lk;
  if (side) {
    side_lk = std::unique_lock<std::mutex>(side->mu);
    MLP_TRY(cuda_err(cudaEventRecord(side->fork, c.stream)));
  }
  if (dx) {
    // dx = s_dpre * s1 * (dP8 W1_8); W1_8 [I,H]: B(n=h, k=i) is N-contiguous
    Gemm g(*p, c.counter(), c.status, pick_cg(M));
    g.p.f8_formats = fmts;
    const int mA = g.kmajor_a_u8(dP8, M, I);
    const int mB = g.mnmajor_u8(W1_8, I, H);
    const int oX = g.output(dx, M, H);
    Prob& P = g.add(M, H, I, 0, MMA_N, 1, 2 * BK);
    P.mapA0 = mA;
    P.mapB0 = mB;
    P.mapO[0] = oX;
    P.sa = scales + 5;  // s_dpre
    P.sb = scales + 1;  // s1
    P.mult = 1.f;
    MLP_TRY((run<EPI_STORE_BF16_F8, false, true>(g, c, MLP_KERNEL_DX)));
  }
  if (want_w) {
    // one grouped launch over the M tokens, both operands MN-major:
    //   dW1 = s_dpre * sx * dP8^T x8  ([I,H])   dW2 = down_mult * sg * s_post * dout8^T a8  ([H,I])
    Call cw = c;
    if (side) {
      cw.stream = side->stream;
      cw.launches = 0;
      MLP_TRY(cuda_err(cudaStreamWaitEvent(side->stream, side->fork, 0)));
    }
    Gemm g(*p, c.counter(), c.status, pick_cg(H < I ? H : I));
    g.p.f8_formats = fmts;
    struct W { const void* A; int rows; const void* B; int cols; void* out; const float* sa;
               const float* sb; float mult; };
    W list[2];
    int n = 0;
    if (dW1) list[n++] = {dP8, I, x8, H, dW1, scales + 5, scales + 0, 1.f};
    if (dW2) list[n++] = {dout8, H, a8, I, dW2, scales + 4, scales + 3, p->down_mult};
    for (int i = 0; i < n; ++i) {
      const int mA = g.mnmajor_u8(list[i].A, M, list[i].rows);
      const int mB = g.mnmajor_u8(list[i].B, M, list[i].cols);
      const int oW = g.output(list[i].out, list[i].rows, list[i].cols);
      Prob& P = g.add(list[i].rows, list[i].cols, M, 0, MMA_N, 1, 2 * BK);
      P.mapA0 = mA;
      P.mapB0 = mB;
      P.mapO[0] = oW;
      P.sa = list[i].sa;
      P.sb = list[i].sb;
      P.mult = list[i].mult;
    }
    MLP_TRY((run<EPI_STORE_BF16_F8, true, true>(g, cw, MLP_KERNEL_WGRAD)));
    if (side) {
      MLP_TRY(cuda_err(cudaEventRecord(side->join, side->stream)));
      MLP_TRY(cuda_err(cudaStreamWaitEvent(c.stream, side->join, 0)));
    }
  }
  return MLP_OK;
}

int mlp_bwd(const mlp_problem_t* p, const void* dout, const void* x, const void* Wg,
            const void* Wu, const void* Wd, void* G, void* U, void* dx, void* dWg, void* dWu,
            void* dWd, int fuse_grad_accum, void* ws, size_t ws_bytes, void* stream) {
  return backward(p, dout, x, Wg, Wu, Wd, G, U, dx, dWg, dWu, dWd, fuse_grad_accum, ws, ws_bytes,
                  stream, false);
}

int mlp_bwd_recompute(const mlp_problem_t* p, const void* dout, const void* x, const void* Wg,
                      const void* Wu, const void* Wd, void* dx, void* dWg, void* dWu, void* dWd,
                      int fuse_grad_accum, void* ws, size_t ws_bytes, void* stream) {
  return backward(p, dout, x, Wg, Wu, Wd, nullptr, nullptr, dx, dWg, dWu, dWd, fuse_grad_accum,
                  ws, ws_bytes, stream, true);
}

int mlp_fp8_refresh_scales(float* amax, float* scale, int n, int width, float gain,
                           float floor_v, void* stream) {
  if (n < 0 || width < 1 || !amax || !scale) return MLP_ERR_INVALID_ARG;
  if (!std::isfinite(gain) || !std::isfinite(floor_v)) return MLP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(amax) & 3u) || (reinterpret_cast<uintptr_t>(scale) & 3u))
    return MLP_ERR_ALIGNMENT;
  if (n == 0) return MLP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return traced(MLP_KERNEL_REFRESH, s, [&] {
    return launch_refresh_scales(amax, scale, n, width, gain, floor_v, s, false);
  });
}

int mlp_plan(const mlp_problem_t* p, int mode, int fuse_grad_accum, mlp_plan_t* plan) {
  if (!plan || check_problem(p) != MLP_OK) return MLP_ERR_INVALID_ARG;
  if (mode < MLP_MODE_FWD || mode > MLP_MODE_FP8_BWD) return MLP_ERR_INVALID_ARG;
  if (fuse_grad_accum != 0 && fuse_grad_accum != 1) return MLP_ERR_INVALID_ARG;
  if (num_sms() <= 0) return MLP_ERR_CUDA;
  std::memset(plan, 0, sizeof(*plan));
  const bool fp8 = mode == MLP_MODE_FP8_FWD || mode == MLP_MODE_FP8_BWD;
  const bool fwd = mode == MLP_MODE_FWD || mode == MLP_MODE_INFER;
  plan->decode = fwd ? decode_kernel(p) : 0;
  plan->cta_group = pick_cg(p->M);
  plan->out_split = (fp8 || plan->decode) ? 1 : out_split_of(p, mode);
  plan->fused_forward = (fwd && !plan->decode && fused_forward(p, plan->out_split)) ? 1 : 0;
  if (!fwd && mode != MLP_MODE_FP8_FWD) {
    const int cg = pick_cg(p->H < p->I ? p->H : p->I);
    long long tiles = out_tiles(p->I, p->H, cg) + out_tiles(p->H, p->I, cg);
    if (gated(p) && !fp8) tiles += out_tiles(p->I, p->H, cg);
    plan->wgrad_cta_group = cg;
    plan->wgrad_split = fp8 ? 1 : wgrad_split(p->M, tiles, cg, fuse_grad_accum);
  }
  return MLP_OK;
}

int mlp_debug_hold_sms(int ctas, unsigned int us, void* stream) {
  if (ctas < 1 || ctas > 65535) return MLP_ERR_INVALID_ARG;
  const unsigned long long ns = (us > 10000000u ? 10000000ull : (unsigned long long)us) * 1000ull;
  return cuda_err(launch_hold(ctas, ns, static_cast<cudaStream_t>(stream)));
}

const char* mlp_status_string(int s) {
  switch (s) {
    case MLP_OK: return "MLP_OK";
    case MLP_ERR_INVALID_ARG: return "MLP_ERR_INVALID_ARG";
    case MLP_ERR_ALIGNMENT: return "MLP_ERR_ALIGNMENT";
    case MLP_ERR_UNSUPPORTED: return "MLP_ERR_UNSUPPORTED";
    case MLP_ERR_WORKSPACE_TOO_SMALL: return "MLP_ERR_WORKSPACE_TOO_SMALL";
    case MLP_ERR_CUDA: return "MLP_ERR_CUDA";
    case MLP_ERR_TIMEOUT: return "MLP_ERR_TIMEOUT";
    default: return "MLP_ERR_UNKNOWN";
  }
}

int mlp_device_status(const void* ws, void* stream) {
  if (!ws) return MLP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MLP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLP_ERR_CUDA;
  return v;
}

const char* mlp_version(void) { return "0.1.0"; }

int mlp_set_tile_policy(int policy) {
  if (policy < 0 || policy > 3) return MLP_ERR_INVALID_ARG;
  g_tile_policy.store(policy);
  return MLP_OK;
}

int mlp_set_wait_timeout_ms(unsigned int ms) {
  g_wait_ms.store(ms);
  return MLP_OK;
}

int mlp_debug_set_flags(int flags) {
  if (flags & ~(MLP_DEBUG_NO_WORK | MLP_DEBUG_DECODE_FMA | MLP_DEBUG_DECODE_MMA))
    return MLP_ERR_INVALID_ARG;
  g_debug_flags.store(flags);
  return MLP_OK;
}

int mlp_trace_enable(int on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = on != 0;
  g_trace_flag.store(g_trace_on);
  return MLP_OK;
}

int mlp_trace_read(int* tags, float* ms, int capacity) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  int n = 0;
  int rc = MLP_OK;
  for (auto& r : g_trace) {
    float t = -1.0f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      rc = MLP_ERR_CUDA;
    if (n < capacity && tags && ms) {
      tags[n] = r.tag;
      ms[n] = t;
    }
    ++n;
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_trace.clear();
  if (rc != MLP_OK) return rc;
  return n < capacity ? n : capacity;
}

const char* mlp_kernel_name(int tag) {
  switch (tag) {
    case MLP_KERNEL_GATE_UP: return "gate_up_act";
    case MLP_KERNEL_DOWN: return "down_proj";
    case MLP_KERNEL_DGATED: return "dgated";
    case MLP_KERNEL_DX: return "dx";
    case MLP_KERNEL_WGRAD: return "wgrad";
    case MLP_KERNEL_POSTACT: return "postact";
    case MLP_KERNEL_CONVERT: return "convert";
    case MLP_KERNEL_DACT_RECOMPUTE: return "dact_recompute";
    case MLP_KERNEL_RSTD: return "rstd";
    case MLP_KERNEL_RMSNORM_BWD: return "rmsnorm_bwd";
    case MLP_KERNEL_QUANT: return "quant_f8";
    case MLP_KERNEL_FWD_FUSED: return "fwd_fused";
    case MLP_KERNEL_REFRESH: return "refresh_scales";
    default: return "unknown";
  }
}

}  // extern "C"
