// gemm.cuh -- the persistent, warp-specialised tcgen05 GEMM with the MLP's
// fused epilogues.
//
// One CTA per SM (320 threads, up to 227 KB shared memory, all 512 TMEM
// columns):
//   warp 0     TMA producer and tile scheduler: fetches work units from a
//              global atomic counter (the first one is the cluster id, except
//              in the one-launch forward), publishes
//              them through a shared-memory ring, and streams the A/B
//              k-blocks of each unit into a ring of as many stages as fit
//              beside the epilogue's staging buffers (six 32 KB stages for
//              a CTA pair, see Cfg).
//   warp 1     allocates TMEM; one lane issues tcgen05.mma (M=128, N=256,
//              K=16) into one of two 256-column fp32 accumulators and
//              commits stage releases / accumulator-full signals.
//   warps 2-9  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//              32*(w%4)..+31, i.e. one output row per thread; warps w and
//              w+4 take the two column halves of those rows), apply the
//              fused activation / derivative / scaling, store to global.
// The double-buffered accumulator lets the epilogue of tile t overlap the
// MMAs of tile t+1.  Every wait is bounded (globaltimer); on expiry the
// kernel records MLP_ERR_TIMEOUT in the status word and unwinds.
// EPI_FWD_FUSED runs the gated forward's two GEMMs in one launch: the
// epilogue warps count their stored gate/up tiles per 256-row block, and the
// producer of a down-projection unit waits for its block's count.
//
// Operand layouts.  A is BM x BK, B is 256 x BK, both bf16 with the
// 128-byte swizzle.  K-major operands ([rows, K], K contiguous) arrive as
// one TMA box {64 (K), rows}; MN-major operands ([K, MN], MN contiguous)
// arrive as boxes {64 (MN), 64 (K)} placed 8 KB apart.  The matching UMMA
// descriptors: K-major SBO = 1024 B (8-row groups), start += 32 B per K=16
// step; MN-major LBO = 8192 B (next 64-wide MN block), SBO = 1024 B (next 8
// K rows), start += 2048 B per K=16 step.  8-bit operands (e4m3 / e5m2)
// keep the 128-byte rows, so a k-block is 128 elements: K-major boxes
// {128 (K), rows} with the same descriptors (+32 B per K=32 step);
// MN-major boxes {128 (MN), 128 (K)} of 16 KB, LBO = 16384 B, SBO = 1024 B,
// start += 4096 B per K=32 step.
#pragma once
#include <atomic>

#include "act.cuh"
#include "gemm_params.h"
#include "ptx.cuh"

namespace mlpk {

constexpr int MLP_ERR_TIMEOUT_CODE = -6;

struct Work {
  int prob, tm, tn, kb_begin, kb_end;
};

__device__ __forceinline__ Work decode_unit(const Params& p, int unit) {
  int pi = 0;
  while (pi + 1 < p.nprob && unit >= p.prob[pi + 1].unit_begin) ++pi;
  const Prob& P = p.prob[pi];
  int u = unit - P.unit_begin;
  int tiles = P.tiles_m * P.tiles_n;
  int ks = u / tiles;
  int t = u - ks * tiles;
  // grouped raster: walk group_m tile rows down a column, then the next column
  const int gm = P.group_m > 0 ? P.group_m : p.group_m;
  int per_group = gm * P.tiles_n;
  int g = t / per_group;
  int first_m = g * gm;
  int gsz = min(P.tiles_m - first_m, gm);
  int r = t - g * per_group;
  Work w;
  w.prob = pi;
  w.tm = first_m + r % gsz;
  w.tn = r / gsz;
  int kb_total = P.kb0 + P.kb1;
  w.kb_begin = ks * P.kper;
  w.kb_end = min(kb_total, w.kb_begin + P.kper);
  return w;
}

// The units of a problem that run the gated forward epilogue.
template <int EPI>
__device__ __forceinline__ bool gated_unit(int prob) {
  return EPI == EPI_GATED_FWD || (EPI == EPI_FWD_FUSED && prob == 0);
}

template <int EPI>
struct EpiTraits {
  // output columns of a tile (EPI_FWD_FUSED: per problem, tile_n_of)
  static constexpr int TILE_N = (EPI == EPI_GATED_FWD) ? 128 : 256;
  // outputs staged per chunk (gated fwd: a, G, U; act fwd: a, P; dgated: dG,
  // dU, a; dact: dP, a; plain: D) and bytes of one staged 32 x 32 box
  static constexpr int NOUT = (EPI == EPI_GATED_FWD || EPI == EPI_DGATED || EPI == EPI_FWD_FUSED) ? 3
                              : (EPI == EPI_ACT_FWD || EPI == EPI_DACT ||
                                 EPI == EPI_DACT_RECOMP || EPI == EPI_ACT_FWD_F8) ? 2
                                                                                  : 1;
  // bytes of a staged 32 x 32 output box: fp32 4096, bf16 2048 (the 8-bit
  // epilogues stage their own boxes, below)
  static constexpr int OUT_BYTES = (EPI == EPI_ACCUM_F32) ? 4096 : 2048;
  // the epilogue reads saved preacts (in0 / in1), fetched ahead of the accumulator
  static constexpr bool DACT = (EPI == EPI_DGATED || EPI == EPI_DACT || EPI == EPI_DGRAD_F8);
  // staged boxes per warp: at most two (a third output reuses the first box
  // once that box's store has read it), so the stage ring keeps 6 stages
  static constexpr int STG_BUFS = NOUT < 2 ? NOUT : 2;
  // 8-bit outputs: the e4m3 postact's 32 x 64-byte half-tile box (+ the bf16
  // preact's chunk box; small enough for a sixth pipeline stage), the e5m2
  // derivative's 32 x 128-byte tile box
  static constexpr int STG_WARP = EPI == EPI_ACT_FWD_F8  ? 2048 + 2048
                                  : (EPI == EPI_DGRAD_F8 || EPI == EPI_DGRAD_F8_RECOMP) ? 4096
                                                        : STG_BUFS * OUT_BYTES;
};

template <int EPI>
__device__ __forceinline__ int tile_n_of(int prob) {
  return gated_unit<EPI>(prob) ? 128 : EpiTraits<EPI>::TILE_N;
}

__device__ __forceinline__ void record_timeout(const Params& p, volatile int* abort_flag) {
  *abort_flag = 1;
  if (p.status) atomicExch(p.status, MLP_ERR_TIMEOUT_CODE);
}

// ---------------------------------------------------------------- epilogues
// Each thread owns one output row of the tile (TMEM lane = row) and walks its
// columns in chunks of 32 (one tcgen05.ld 32x32b.x32).  A warp's 32 rows x
// 32 columns of each output are staged in shared memory and written with
// one TMA store per output: bf16 boxes (64 B rows) use the 64-byte swizzle,
// fp32 boxes (128 B rows) the 128-byte swizzle, so that the row-per-thread
// 16-byte shared stores are free of bank conflicts.  TMA clips the boxes at
// the tensor's edges.  tcgen05.ld is warp-collective, so every lane issues
// it whatever its row's validity.

struct EpiWarp {
  uint32_t stg;  // this warp's staging buffers
  int lane;
  int row0;      // first of the warp's 32 rows
  bool rows_ok;  // any of the 32 rows inside the output
  uint32_t box;  // EPI_DACT_RECOMP: which of the two boxes the next chunk fills
  float rs;      // this lane's row scale (the block's RMS norm; 1 without it)
  // EPI_DGRAD_F8 with TMA-loaded preact boxes: the two halves of the staging
  // box each have a barrier (ebar, ebar + 8); ephase holds their parities,
  // epend the halves with a load in flight (bit per half)
  uint32_t ebar;
  uint32_t ephase;
  uint32_t epend;
};

// Stage this lane's 32 bf16 (16 packed words) into a 64B-swizzled 32x32 box.
__device__ __forceinline__ void stage_bf16(uint32_t buf, int r, const uint32_t (&w)[16]) {
  const uint32_t rb = buf + static_cast<uint32_t>(r) * 64u;
  const uint32_t x = (static_cast<uint32_t>(r) >> 1) & 3u;
#pragma unroll
  for (uint32_t j = 0; j < 4; ++j)
    st_shared_v4(rb + ((j ^ x) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

// Stage this lane's 32 fp32 values into a 128B-swizzled 32x32 box.
__device__ __forceinline__ void stage_f32(uint32_t buf, int r, const uint32_t (&w)[32]) {
  const uint32_t rb = buf + static_cast<uint32_t>(r) * 128u;
  const uint32_t x = static_cast<uint32_t>(r) & 7u;
#pragma unroll
  for (uint32_t j = 0; j < 8; ++j)
    st_shared_v4(rb + ((j ^ x) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

// What the epilogue needs of a work unit's problem, read from the launch
// parameters once per unit and kept in registers (a per-chunk read would be
// a generic load re-issued after every store's memory clobber).
struct EpiUnit {
  const CUtensorMap* out[3];  // output maps (nullptr: output not written)
  int M, N, ld;
  const void* in0;            // saved preacts (derivative epilogues); the residual (plain store)
  const void* in1;
  const float* rstd;          // per-row scale (nullptr: none)
  float alpha;                // residual scale
  float deq;                  // 8-bit epilogues: *sa * *sb (the operands' dequant scales)
  float deq0;                 // ... EPI_DGRAD_F8_RECOMP: *sp0 * *sp1 (the recomputed preact's)
  float mult;                 // ... the problem's multiplier
  float inv;                  // ... fp32(1 / *sq), the 8-bit output's quantisation factor
  float* amax;                // running max of the 8-bit epilogue's output
  const CUtensorMap* ein;     // EPI_DGRAD_F8: in0's 32 x 32 boxes for TMA loads (nullptr: none)
};

// deq, inv: the 8-bit epilogues' factors of this problem (read once per kernel)
template <int EPI>
__device__ __forceinline__ EpiUnit epi_unit(const Params& p, const Prob& P, float deq, float inv,
                                            float deq0 = 1.f) {
  EpiUnit U;
#pragma unroll
  for (int o = 0; o < 3; ++o) U.out[o] = P.mapO[o] >= 0 ? &p.maps[P.mapO[o]] : nullptr;
  U.M = P.M;
  U.N = P.N;
  U.ld = P.ld;
  U.in0 = P.in0;
  U.in1 = P.in1;
  U.rstd = P.rstd;
  U.alpha = P.alpha;
  U.deq = 1.f;
  U.mult = 1.f;
  U.inv = 1.f;
  U.amax = nullptr;
  U.ein = P.mapE >= 0 ? &p.maps[P.mapE] : nullptr;
  U.deq0 = 1.f;
  if constexpr (is_f8(EPI)) {
    U.deq = deq;
    U.deq0 = deq0;
    U.mult = P.mult;
    U.inv = inv;
    U.amax = P.amax;
  }
  return U;
}

// The staging buffers may be overwritten once the previous chunk's stores
// have read them.
__device__ __forceinline__ void staging_acquire(const EpiWarp& e) {
  if (e.lane == 0) bulk_wait_read_all();
  __syncwarp();
}

// Store the staged boxes of outputs whose map exists at (col, row0).
template <int NOUT, int OUT_BYTES, bool REDUCE>
__device__ __forceinline__ void flush_chunk(const Params& p, const EpiUnit& P, const EpiWarp& e,
                                            int col) {
  fence_proxy_async_smem();
  __syncwarp();
  if (e.lane == 0) {
#pragma unroll
    for (int o = 0; o < NOUT; ++o) {
      if (P.out[o]) {
        const CUtensorMap* m = P.out[o];
        if constexpr (REDUCE) tma_reduce_add_2d(m, e.stg + o * OUT_BYTES, col, e.row0);
        else tma_store_2d(m, e.stg + o * OUT_BYTES, col, e.row0);
      }
    }
    bulk_commit();
  }
}

// Store staged box `buf` of output o (if its map exists) as a bulk group of its own.
__device__ __forceinline__ void store_box(const Params& p, const EpiUnit& P, const EpiWarp& e, int o,
                                          uint32_t buf, int col) {
  fence_proxy_async_smem();
  __syncwarp();
  if (e.lane == 0) {
    if (P.out[o]) tma_store_2d(P.out[o], buf, col, e.row0);
    bulk_commit();
  }
}

// Wait until all but the newest of this warp's bulk store groups have read
// their boxes (the oldest box may then be refilled).
__device__ __forceinline__ void staging_wait_read_but_one(const EpiWarp& e) {
  if (e.lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
  __syncwarp();
}

template <int ACT>
__device__ __forceinline__ void epi_gated_fwd(const Params& p, const EpiUnit& P, const EpiWarp& e,
                                              uint32_t tb, int col0, int cb, int ce) {
  const float s = p.scale;
#pragma unroll 1
  for (int c = cb; c < ce; c += 32) {
    const int col = col0 + c;
    if (col >= P.N) break;  // warp-uniform
    uint32_t g[32], u[32];
    __syncwarp();
    tmem_ld32(tb + c, g);
    tmem_ld32(tb + 128 + c, u);
    tmem_wait_ld();
    uint32_t pa[16], pg[16], pu[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      // the block's RMS norm of the input row, applied to the preacts
      const float g0 = e.rs * __uint_as_float(g[2 * j]), g1 = e.rs * __uint_as_float(g[2 * j + 1]);
      const float u0 = e.rs * __uint_as_float(u[2 * j]), u1 = e.rs * __uint_as_float(u[2 * j + 1]);
      pa[j] = pack_bf16x2(s * act_f<ACT>(g0) * u0, s * act_f<ACT>(g1) * u1);
      pg[j] = pack_bf16x2(g0, g1);
      pu[j] = pack_bf16x2(u0, u1);
    }
    // a and G through the two boxes, then U through the first again
    staging_acquire(e);
    stage_bf16(e.stg, e.lane, pa);
    if (P.out[1]) stage_bf16(e.stg + 2048, e.lane, pg);
    store_box(p, P, e, 0, e.stg, col);
    store_box(p, P, e, 1, e.stg + 2048, col);
    if (P.out[2]) {
      staging_wait_read_but_one(e);
      stage_bf16(e.stg, e.lane, pu);
      store_box(p, P, e, 2, e.stg, col);
    }
  }
}

template <int ACT>
__device__ __forceinline__ void epi_act_fwd(const Params& p, const EpiUnit& P, const EpiWarp& e,
                                            uint32_t tb, int col0, int cb, int ce) {
  const float s = p.scale;
#pragma unroll 1
  for (int c = cb; c < ce; c += 32) {
    const int col = col0 + c;
    if (col >= P.N) break;
    uint32_t z[32];
    __syncwarp();
    tmem_ld32(tb + c, z);
    tmem_wait_ld();
    uint32_t pa[16], pp[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float z0 = e.rs * __uint_as_float(z[2 * j]), z1 = e.rs * __uint_as_float(z[2 * j + 1]);
      pa[j] = pack_bf16x2(s * act_f<ACT>(z0), s * act_f<ACT>(z1));
      pp[j] = pack_bf16x2(z0, z1);
    }
    staging_acquire(e);
    stage_bf16(e.stg, e.lane, pa);
    if (P.out[1]) stage_bf16(e.stg + 2048, e.lane, pp);
    flush_chunk<2, 2048, false>(p, P, e, col);
  }
}

// Loads this thread's 32 saved preacts (G and, if gated, U) of chunk `col`.
template <bool GATED>
__device__ __forceinline__ void dact_load(const EpiUnit& P, int row, int col, uint4 (&g)[4],
                                          uint4 (&u)[4]) {
  const __nv_bfloat16* g_in = static_cast<const __nv_bfloat16*>(P.in0);
  const __nv_bfloat16* u_in = static_cast<const __nv_bfloat16*>(P.in1);
  const bool row_ok = row < P.M;
  const size_t off = static_cast<size_t>(row) * P.ld + col;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const bool ok = row_ok && (col + 8 * v < P.N);
    g[v] = ok ? ld_global_v4(g_in + off + 8 * v) : make_uint4(0, 0, 0, 0);
    u[v] = (GATED && ok) ? ld_global_v4(u_in + off + 8 * v) : make_uint4(0, 0, 0, 0);
  }
}

// The same preacts, read row-coalesced: load i of lane l holds columns
// col + 8 (l % 4) .. + 7 of row row0 + 8 i + l / 4, so each load of the warp
// reads eight 64-byte row pieces instead of 32 16-byte ones.
// dact_rows_to_lanes then gives each lane its own row.
template <bool GATED>
__device__ __forceinline__ void dact_load_rows(const EpiUnit& P, int row0, int lane, int col,
                                               uint4 (&g)[4], uint4 (&u)[4]) {
  const __nv_bfloat16* g_in = static_cast<const __nv_bfloat16*>(P.in0);
  const __nv_bfloat16* u_in = static_cast<const __nv_bfloat16*>(P.in1);
  const int v = lane & 3;
  const bool col_ok = col + 8 * v < P.N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = row0 + 8 * i + (lane >> 2);
    const bool ok = col_ok && row < P.M;
    const size_t off = static_cast<size_t>(row) * P.ld + col + 8 * v;
    g[i] = ok ? ld_global_v4(g_in + off) : make_uint4(0, 0, 0, 0);
    u[i] = (GATED && ok) ? ld_global_v4(u_in + off) : make_uint4(0, 0, 0, 0);
  }
}

// From dact_load_rows' order to this lane's row (g[v], u[v]: columns 8v ..
// 8v + 7 of row `lane`), through the warp's staging boxes (G in the first,
// U in the second; 64-byte rows, 16-byte units swizzled by (row / 2) % 4, so
// neither the row-order writes nor the row-per-lane reads conflict).  The
// boxes must be free (staging_acquire); each lane's outputs later overwrite
// only the row it has read.
template <bool GATED>
__device__ __forceinline__ void dact_rows_to_lanes(const EpiWarp& e, uint4 (&g)[4], uint4 (&u)[4]) {
  const uint32_t lane = static_cast<uint32_t>(e.lane);
#pragma unroll
  for (uint32_t i = 0; i < 4; ++i) {
    const uint32_t r = 8u * i + (lane >> 2), v = lane & 3u;
    const uint32_t a = r * 64u + ((v ^ ((r >> 1) & 3u)) << 4);
    st_shared_v4(e.stg + a, g[i].x, g[i].y, g[i].z, g[i].w);
    if (GATED) st_shared_v4(e.stg + 2048 + a, u[i].x, u[i].y, u[i].z, u[i].w);
  }
  __syncwarp();
  const uint32_t x = (lane >> 1) & 3u;
#pragma unroll
  for (uint32_t v = 0; v < 4; ++v) {
    const uint32_t a = lane * 64u + ((v ^ x) << 4);
    g[v] = ld_shared_v4(e.stg + a);
    if (GATED) u[v] = ld_shared_v4(e.stg + 2048 + a);
  }
}

// GATED = true: in0 = G, in1 = U -> outputs dG, dU, a (maps 0, 1, 2)
// GATED = false: in0 = P -> outputs dP, a (maps 0, 1)
// The saved preacts of chunk c+1 are loaded (row-coalesced, dact_load_rows)
// while chunk c is computed; the caller has already loaded chunk `cb` into
// (pg, pu) before waiting for the accumulator.  Each chunk's preacts pass
// through the staging boxes to one row per lane before its outputs are
// staged there (measured back to back, two builds, outputs bitwise equal:
// 2.7-3.3 % off the derivative GEMM on the 4096- and 2048-wide SwiGLU
// shapes, 2.8 % off the ReLU^2 backward, Llama-3-8B's unchanged).  In-place
// outputs are safe: every element is read (global load) before the TMA
// store of its chunk is issued, and chunks do not overlap.
template <int ACT, bool GATED>
__device__ __forceinline__ void epi_dact(const Params& p, const EpiUnit& P, const EpiWarp& e,
                                         uint32_t tb, int col0, int cb, int ce, uint4 (&pg)[4],
                                         uint4 (&pu)[4]) {
  const float s = p.scale;
  const float sr = s * e.rs;
  constexpr int NOUT = GATED ? 3 : 2;
#pragma unroll 1
  for (int c = cb; c < ce; c += 32) {
    const int col = col0 + c;
    if (col >= P.N) break;
    uint4 ng[4], nu[4];
    if (c + 32 < ce) dact_load_rows<GATED>(P, e.row0, e.lane, col + 32, ng, nu);
    uint32_t d[32];
    __syncwarp();
    tmem_ld32(tb + c, d);
    tmem_wait_ld();
    // dG (dP) to the first box and dU (gated) or the postact (non-gated) to
    // the second, one 8-column group at a time; a gated postact waits in
    // registers for the first box to be read, then goes out through it
    staging_acquire(e);
    dact_rows_to_lanes<GATED>(e, pg, pu);
    const bool want_a = P.out[NOUT - 1] != nullptr;
    const uint32_t rb = static_cast<uint32_t>(e.lane) * 64u;
    const uint32_t x = (static_cast<uint32_t>(e.lane) >> 1) & 3u;
    uint32_t pa[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint32_t gw[4] = {pg[v].x, pg[v].y, pg[v].z, pg[v].w};
      const uint32_t uw[4] = {pu[v].x, pu[v].y, pu[v].z, pu[v].w};
      uint32_t pdg[4], pdu[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 gg = unpack_bf16x2(gw[j]);
        if constexpr (GATED && ACT == ACT_SILU) {
          // SwiGLU: the arithmetic below (and act_and_grad's) two lanes at a
          // time in fp32x2 instructions; each lane rounds as the scalar code
          // would, so the results are bitwise the same (measured 1.5-2 % off
          // dgated's time)
          {  // (scope of the packed temporaries)
            const uint64_t half2 = f2_pack(0.5f, 0.5f), one2 = f2_pack(1.f, 1.f);
            const uint64_t g2 = f2_pack(gg.x, gg.y);
            const float2 uu = unpack_bf16x2(uw[j]);
            const uint64_t u2 = f2_pack(uu.x, uu.y);
            const uint64_t dh = f2_mul(f2_pack(sr, sr), f2_pack(__uint_as_float(d[8 * v + 2 * j]),
                                                                __uint_as_float(d[8 * v + 2 * j + 1])));
            const float2 h = f2_unpack(f2_mul(half2, g2));
            const uint64_t sg = f2_fma(half2, f2_pack(tanh_hw(h.x), tanh_hw(h.y)), half2);
            const uint64_t a2 = f2_mul(g2, sg);
            const uint64_t da2 =
                f2_mul(sg, f2_fma(g2, f2_fma(f2_pack(-1.f, -1.f), sg, one2), one2));
            const float2 dg = f2_unpack(f2_mul(f2_mul(dh, u2), da2));
            const float2 du = f2_unpack(f2_mul(dh, a2));
            const float2 pv = f2_unpack(f2_mul(f2_mul(f2_pack(s, s), a2), u2));
            pdg[j] = pack_bf16x2(dg.x, dg.y);
            pdu[j] = pack_bf16x2(du.x, du.y);
            pa[4 * v + j] = pack_bf16x2(pv.x, pv.y);
            continue;
          }
        }
        // (times the row scale of the block's RMS norm: the weight and input
        // gradients then come out in terms of the un-normalised input)
        const float dh0 = sr * __uint_as_float(d[8 * v + 2 * j]);
        const float dh1 = sr * __uint_as_float(d[8 * v + 2 * j + 1]);
        float a0, da0, a1, da1;
        act_and_grad<ACT>(gg.x, a0, da0);
        act_and_grad<ACT>(gg.y, a1, da1);
        if (GATED) {
          const float2 uu = unpack_bf16x2(uw[j]);
          pdg[j] = pack_bf16x2(dh0 * uu.x * da0, dh1 * uu.y * da1);
          pdu[j] = pack_bf16x2(dh0 * a0, dh1 * a1);
          pa[4 * v + j] = pack_bf16x2(s * a0 * uu.x, s * a1 * uu.y);
        } else {
          pdg[j] = pack_bf16x2(dh0 * da0, dh1 * da1);
          pa[4 * v + j] = pack_bf16x2(s * a0, s * a1);
        }
      }
      const uint32_t unit = rb + ((static_cast<uint32_t>(v) ^ x) << 4);
      st_shared_v4(e.stg + unit, pdg[0], pdg[1], pdg[2], pdg[3]);
      if (GATED) {
        st_shared_v4(e.stg + 2048 + unit, pdu[0], pdu[1], pdu[2], pdu[3]);
      } else if (want_a) {
        st_shared_v4(e.stg + 2048 + unit, pa[4 * v], pa[4 * v + 1], pa[4 * v + 2], pa[4 * v + 3]);
      }
    }
    store_box(p, P, e, 0, e.stg, col);
    store_box(p, P, e, 1, e.stg + 2048, col);  // dU, or the non-gated postact
    if (GATED && want_a) {
      staging_wait_read_but_one(e);
      stage_bf16(e.stg, e.lane, pa);
      store_box(p, P, e, 2, e.stg, col);
    }
    if (c + 32 < ce) {
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        pg[v] = ng[v];
        pu[v] = nu[v];
      }
    }
  }
}

// Fused recompute + derivative (non-gated), in two phases per tile.  Every
// chunk is one 32 x 32 bf16 box; the two staging boxes alternate across
// chunks, phases and tiles (e.box), so a box is refilled once every store
// group but the newest has read its box.
//
// Phase 1, accumulator p = x W1^T: the postact a = s*act(p) goes out
// through map 1 (if requested); s*act'(p) of the thread's 128 columns stays
// in registers as packed bf16 pairs (dd; 128 fp32 values would not fit the
// 168 registers a thread of this kernel gets), the same rounding the
// unfused path takes when it stores P in bf16, and the accumulator is
// handed back to the MMAs, which compute the next p while phase 2 runs.
template <int ACT>
__device__ __forceinline__ void epi_recomp_p(const Params& p, const EpiUnit& P, EpiWarp& e,
                                             uint32_t tb, int col0, int cb, uint32_t (&dd)[64]) {
  const float s = p.scale;
  const bool want_a = P.out[1] != nullptr;
#pragma unroll
  for (int ci = 0; ci < 4; ++ci) {
    const int c = cb + 32 * ci;
    const int col = col0 + c;
    if (col >= P.N) break;  // warp-uniform
    uint32_t z[32];
    __syncwarp();
    tmem_ld32(tb + c, z);
    tmem_wait_ld();
    uint32_t pa[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float a0, a1, d0, d1;
      act_and_grad<ACT>(__uint_as_float(z[2 * j]), a0, d0);
      act_and_grad<ACT>(__uint_as_float(z[2 * j + 1]), a1, d1);
      dd[16 * ci + j] = pack_bf16x2(s * d0, s * d1);
      pa[j] = pack_bf16x2(s * a0, s * a1);
    }
    if (want_a) {
      const uint32_t buf = e.stg + e.box * 2048u;
      staging_wait_read_but_one(e);
      stage_bf16(buf, e.lane, pa);
      store_box(p, P, e, 1, buf, col);
      e.box ^= 1u;
    }
  }
}

// Phase 2, accumulator dh = dout Wd: dP = dh * s*act'(p) through map 0.
__device__ __forceinline__ void epi_recomp_dh(const Params& p, const EpiUnit& P, EpiWarp& e,
                                              uint32_t tb, int col0, int cb,
                                              const uint32_t (&dd)[64]) {
#pragma unroll
  for (int ci = 0; ci < 4; ++ci) {
    const int c = cb + 32 * ci;
    const int col = col0 + c;
    if (col >= P.N) break;
    uint32_t d[32];
    __syncwarp();
    tmem_ld32(tb + c, d);
    tmem_wait_ld();
    uint32_t q[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float2 g = unpack_bf16x2(dd[16 * ci + j]);
      q[j] = pack_bf16x2(__uint_as_float(d[2 * j]) * g.x, __uint_as_float(d[2 * j + 1]) * g.y);
    }
    const uint32_t buf = e.stg + e.box * 2048u;
    staging_wait_read_but_one(e);
    stage_bf16(buf, e.lane, q);
    store_box(p, P, e, 0, buf, col);
    e.box ^= 1u;
  }
}

// 8-bit outputs are staged a whole tile row block at a time: the warp's 32
// rows x 128 columns (one byte each) in one 32 x 128-byte box with the
// 128-byte swizzle (16-byte unit u of row r at unit u ^ (r % 8): a warp's
// row-per-thread 16-byte stores are conflict-free), stored by one TMA store
// per tile.  Lane r writes bytes [32 c, 32 c + 32) of its row for chunk c.
__device__ __forceinline__ void stage_f8_chunk(uint32_t buf, int r, int c, const uint32_t (&q)[8]) {
  const uint32_t rb = buf + static_cast<uint32_t>(r) * 128u;
  const uint32_t x = static_cast<uint32_t>(r) & 7u;
  const uint32_t u = 2u * static_cast<uint32_t>(c);
  st_shared_v4(rb + ((u ^ x) << 4), q[0], q[1], q[2], q[3]);
  st_shared_v4(rb + (((u + 1u) ^ x) << 4), q[4], q[5], q[6], q[7]);
}

// The same for a 32 x 64-byte box with the 64-byte swizzle (16-byte unit u
// of row r at unit u ^ ((r / 2) % 4)): lane r writes bytes [32 h, 32 h + 32)
// of its row for the box's chunk h (0 or 1).
__device__ __forceinline__ void stage_f8_half(uint32_t buf, int r, int h, const uint32_t (&q)[8]) {
  const uint32_t rb = buf + static_cast<uint32_t>(r) * 64u;
  const uint32_t x = (static_cast<uint32_t>(r) >> 1) & 3u;
  const uint32_t u = 2u * static_cast<uint32_t>(h);
  st_shared_v4(rb + ((u ^ x) << 4), q[0], q[1], q[2], q[3]);
  st_shared_v4(rb + (((u + 1u) ^ x) << 4), q[4], q[5], q[6], q[7]);
}

// Store the staged 8-bit box of output o at (col, row0) as a bulk group.
__device__ __forceinline__ void store_f8_tile(const EpiUnit& P, const EpiWarp& e, int o,
                                              uint32_t buf, int col) {
  fence_proxy_async_smem();
  __syncwarp();
  if (e.lane == 0) {
    if (P.out[o]) tma_store_2d(P.out[o], buf, col, e.row0);
    bulk_commit();
  }
}

// e4m3 forward of the ReLU^2 MLP: pre = acc * sx * s1, a = mult * relu(pre)^2,
// a -> e4m3(a * fp32(1 / s_post)) (map 0, staged two chunks at a time in a
// 32 x 64-byte box at stg) and, if requested, pre in bf16 through a 32 x 32
// bf16 box per chunk (map 1, at stg + 2048; for the backward); the largest
// |a| of the warp's rows goes to *amax (atomic max on the bits of a
// non-negative float).
template <int ACT>
__device__ __forceinline__ void epi_act_f8(const Params& p, const EpiUnit& P, const EpiWarp& e,
                                           uint32_t tb, int col0, int cb, int ce) {
  const float deq = P.deq;
  const float inv = P.inv;
  const float s = P.mult;
  const bool want_pre = P.out[1] != nullptr;
  const bool row_ok = e.row0 + e.lane < P.M;
  const uint32_t pbuf = e.stg + 2048u;
  float mx = 0.f;
#pragma unroll 1
  for (int c = cb; c < ce; c += 32) {
    const int col = col0 + c;
    if (col >= P.N) break;
    uint32_t z[32];
    __syncwarp();
    tmem_ld32(tb + c, z);
    tmem_wait_ld();
    uint32_t q[8], pp[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t w = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int k = 4 * j + 2 * h;
        const float z0 = __uint_as_float(z[k]) * deq, z1 = __uint_as_float(z[k + 1]) * deq;
        pp[2 * j + h] = pack_bf16x2(z0, z1);
        const float p0 = fmaxf(z0, 0.f), p1 = fmaxf(z1, 0.f);
        const float a0 = s * p0 * p0, a1 = s * p1 * p1;
        mx = fmaxf(mx, fmaxf(fabsf(a0), fabsf(a1)));
        w |= static_cast<uint32_t>(pack_e4m3x2(a0 * inv, a1 * inv)) << (16 * h);
      }
      q[j] = w;
    }
    // the previous chunk's preact box (and the last stored code box) must
    // have been read before they are overwritten
    staging_acquire(e);
    const int k = (c - cb) >> 5;  // chunk of the warp's columns
    stage_f8_half(e.stg, e.lane, k & 1, q);
    if (want_pre) {
      stage_bf16(pbuf, e.lane, pp);
      store_box(p, P, e, 1, pbuf, col);
    }
    // a code box goes out once both of its chunks are staged, or after the
    // warp's last chunk (TMA clips it at the output's edge)
    if ((k & 1) || c + 32 >= ce || col + 32 >= P.N) store_f8_tile(P, e, 0, e.stg, col - 32 * (k & 1));
  }
  if (P.amax) {
    if (!row_ok) mx = 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (e.lane == 0 && mx > 0.f) atomicMax(reinterpret_cast<int*>(P.amax), __float_as_int(mx));
  }
}

// e5m2 derivative of the 8-bit ReLU^2 MLP: dpre = deq * acc * 2 * relu(P)
// with P the saved bf16 preact (in0), dpre -> e5m2(dpre * fp32(1 / *sq))
// (map 0, staged per tile); the largest |dpre| of the warp's rows goes to
// *amax.  The caller loads P's first chunk before waiting for the
// accumulator; the other three chunks of the tile are loaded here before the
// first is used (the producer has prefetched the tile into L2).
__device__ __forceinline__ void epi_dgrad_f8(const Params& p, const EpiUnit& P, const EpiWarp& e,
                                             uint32_t tb, int col0, int cb, int ce,
                                             uint4 (&pg)[4]) {
  const float dq2 = 2.f * P.mult * P.deq;
  const float inv = P.inv;
  const int row = e.row0 + e.lane;
  uint4 pr[3][4], unused[4];
#pragma unroll
  for (int i = 0; i < 3; ++i) dact_load<false>(P, row, col0 + cb + 32 * (i + 1), pr[i], unused);
  float mx = 0.f;
#pragma unroll
  for (int ci = 0; ci < 4; ++ci) {
    const int col = col0 + cb + 32 * ci;
    if (col >= P.N) break;
    uint32_t z[32];
    __syncwarp();
    tmem_ld32(tb + cb + 32 * ci, z);
    tmem_wait_ld();
    uint32_t q[8];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 g4 = ci == 0 ? pg[v] : pr[ci - 1][v];
      const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
      q[2 * v] = 0;
      q[2 * v + 1] = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 pv = unpack_bf16x2(gw[j]);
        const float d0 = dq2 * __uint_as_float(z[8 * v + 2 * j]) * fmaxf(pv.x, 0.f);
        const float d1 = dq2 * __uint_as_float(z[8 * v + 2 * j + 1]) * fmaxf(pv.y, 0.f);
        mx = fmaxf(mx, fmaxf(fabsf(d0), fabsf(d1)));
        q[2 * v + (j >> 1)] |= static_cast<uint32_t>(pack_e5m2x2(d0 * inv, d1 * inv))
                               << (16 * (j & 1));
      }
    }
    if (ci == 0) staging_acquire(e);  // the previous tile's box has been read
    stage_f8_chunk(e.stg, e.lane, ci, q);
  }
  if (col0 + cb < P.N) store_f8_tile(P, e, 0, e.stg, col0 + cb);
  if (P.amax) {
    if (row >= P.M) mx = 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (e.lane == 0 && mx > 0.f) atomicMax(reinterpret_cast<int*>(P.amax), __float_as_int(mx));
  }
}

// EPI_DGRAD_F8 with the saved preact loaded by TMA (P.ein).  Loading P row
// by row (each lane its own row's 64 bytes a chunk) costs a warp 32 L1
// wavefronts per 16-byte load and was the largest part of this epilogue.
// Instead the warp's 4 KB staging box serves as two 2 KB buffers, X (stg)
// and Y (stg + 2048), that take P's 32 x 32 bf16 boxes (64-byte swizzle):
// chunks 0 and 2 in X, 1 and 3 in Y, each with its own barrier.  The e5m2
// codes of a chunk stay in registers (8 a lane) until the tile's last chunk
// is done; the box then stages them for the one TMA store per tile.
//
// dgrad_f8_issue: the loads of chunks 0 and 1 of a tile, issued before the
// wait for the accumulator (the previous tile's store must have read the
// box first).
__device__ __forceinline__ void dgrad_f8_issue(const EpiUnit& P, EpiWarp& e, int col, int half,
                                               uint64_t pol) {
  if (col >= P.N) return;  // warp-uniform
  e.epend |= 1u << half;
  if (e.lane == 0) {
    const uint32_t bar = e.ebar + 8u * static_cast<uint32_t>(half);
    mbar_expect_tx(bar, 2048);
    tma_load_2d(e.stg + 2048u * static_cast<uint32_t>(half), P.ein, col, e.row0, bar, pol);
  }
}

// After an expired wait: let the loads still in flight land (bounded)
// before the kernel unwinds and its shared memory is released.
__device__ __forceinline__ void dgrad_f8_drain(EpiWarp& e) {
  volatile int never = 0;
#pragma unroll
  for (uint32_t h = 0; h < 2; ++h) {
    if (e.epend & (1u << h)) {
      mbar_wait(e.ebar + 8u * h, (e.ephase >> h) & 1u, 10000000ull, &never);
      e.ephase ^= 1u << h;
    }
  }
  e.epend = 0;
}

// The tile's epilogue; false when a bounded wait expired (loads drained).
__device__ __forceinline__ bool epi_dgrad_f8_tma(const EpiUnit& P, EpiWarp& e, uint32_t tb,
                                                 int col0, int cb, uint64_t lim,
                                                 volatile int* abort_flag, uint64_t pol) {
  const float dq2 = 2.f * P.mult * P.deq;
  const float inv = P.inv;
  const int row = e.row0 + e.lane;
  const uint32_t rb = static_cast<uint32_t>(e.lane) * 64u;
  const uint32_t x = (static_cast<uint32_t>(e.lane) >> 1) & 3u;
  uint32_t qq[4][8];
  float mx = 0.f;
  int nch = 0;
#pragma unroll
  for (int ci = 0; ci < 4; ++ci) {
    const int col = col0 + cb + 32 * ci;
    if (col >= P.N) break;  // warp-uniform
    const uint32_t h = static_cast<uint32_t>(ci & 1);
    const uint32_t buf = e.stg + 2048u * h;
    if (!mbar_wait(e.ebar + 8u * h, (e.ephase >> h) & 1u, lim, abort_flag)) {
      dgrad_f8_drain(e);
      return false;
    }
    e.ephase ^= 1u << h;
    e.epend &= ~(1u << h);
    // this lane's row of the chunk (16-byte unit u sits at u ^ ((r / 2) % 4))
    uint4 pv[4];
#pragma unroll
    for (uint32_t v = 0; v < 4; ++v) pv[v] = ld_shared_v4(buf + rb + ((v ^ x) << 4));
    uint32_t z[32];
    __syncwarp();
    tmem_ld32(tb + cb + 32 * ci, z);
    tmem_wait_ld();
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint32_t gw[4] = {pv[v].x, pv[v].y, pv[v].z, pv[v].w};
      qq[ci][2 * v] = 0;
      qq[ci][2 * v + 1] = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 pp = unpack_bf16x2(gw[j]);
        const float d0 = dq2 * __uint_as_float(z[8 * v + 2 * j]) * fmaxf(pp.x, 0.f);
        const float d1 = dq2 * __uint_as_float(z[8 * v + 2 * j + 1]) * fmaxf(pp.y, 0.f);
        mx = fmaxf(mx, fmaxf(fabsf(d0), fabsf(d1)));
        qq[ci][2 * v + (j >> 1)] |= static_cast<uint32_t>(pack_e5m2x2(d0 * inv, d1 * inv))
                                    << (16 * (j & 1));
      }
    }
    nch = ci + 1;
    // every lane has used its row of the buffer (the codes above depend on
    // it): chunk ci + 2 may go there
    __syncwarp();
    if (ci < 2) {
      if (e.lane == 0) fence_proxy_async_smem();
      dgrad_f8_issue(P, e, col + 64, static_cast<int>(h), pol);
    }
  }
  // every load issued for this tile has been waited for: the box is free
#pragma unroll
  for (int ci = 0; ci < 4; ++ci)
    if (ci < nch) stage_f8_chunk(e.stg, e.lane, ci, qq[ci]);
  if (nch > 0) store_f8_tile(P, e, 0, e.stg, col0 + cb);
  if (P.amax) {
    if (row >= P.M) mx = 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (e.lane == 0 && mx > 0.f) atomicMax(reinterpret_cast<int*>(P.amax), __float_as_int(mx));
  }
  return true;
}

// EPI_DGRAD_F8_RECOMP, phase 1 on accumulator 0 (x8 W1_8^T): this thread's
// 128 values of dd = 2 relu(deq0 * acc) as packed bf16 pairs (the saved-
// preact path's 2 relu(bf16(pre)): doubling and relu commute with the
// rounding), after which the accumulator goes back to the MMAs.
__device__ __forceinline__ void epi_recomp_f8_p(const EpiUnit& P, uint32_t tb, int col0, int cb,
                                                uint32_t (&dd)[64]) {
  const float deq0 = P.deq0;
#pragma unroll
  for (int ci = 0; ci < 4; ++ci) {
    const int c = cb + 32 * ci;
    if (col0 + c >= P.N) break;  // warp-uniform
    uint32_t z[32];
    __syncwarp();
    tmem_ld32(tb + c, z);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float r0 = fmaxf(deq0 * __uint_as_float(z[2 * j]), 0.f);
      const float r1 = fmaxf(deq0 * __uint_as_float(z[2 * j + 1]), 0.f);
      dd[16 * ci + j] = pack_bf16x2(2.f * r0, 2.f * r1);
    }
  }
}

// Phase 2 on accumulator 1 (dout8 W2_8): dpre = mult * deq * acc * dd ->
// e5m2(dpre * fp32(1 / *sq)) staged per tile as in epi_dgrad_f8; the largest
// |dpre| of the warp's rows goes to *amax.
__device__ __forceinline__ void epi_recomp_f8_dh(const EpiUnit& P, const EpiWarp& e, uint32_t tb,
                                                 int col0, int cb, const uint32_t (&dd)[64]) {
  const float dq = P.mult * P.deq;
  const float inv = P.inv;
  float mx = 0.f;
#pragma unroll
  for (int ci = 0; ci < 4; ++ci) {
    const int col = col0 + cb + 32 * ci;
    if (col >= P.N) break;
    uint32_t z[32];
    __syncwarp();
    tmem_ld32(tb + cb + 32 * ci, z);
    tmem_wait_ld();
    uint32_t q[8];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      q[2 * v] = 0;
      q[2 * v + 1] = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 g = unpack_bf16x2(dd[16 * ci + 4 * v + j]);
        const float d0 = dq * __uint_as_float(z[8 * v + 2 * j]) * g.x;
        const float d1 = dq * __uint_as_float(z[8 * v + 2 * j + 1]) * g.y;
        mx = fmaxf(mx, fmaxf(fabsf(d0), fabsf(d1)));
        q[2 * v + (j >> 1)] |= static_cast<uint32_t>(pack_e5m2x2(d0 * inv, d1 * inv))
                               << (16 * (j & 1));
      }
    }
    if (ci == 0) staging_acquire(e);  // the previous tile's box has been read
    stage_f8_chunk(e.stg, e.lane, ci, q);
  }
  if (col0 + cb < P.N) store_f8_tile(P, e, 0, e.stg, col0 + cb);
  if (P.amax) {
    if (e.row0 + e.lane >= P.M) mx = 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (e.lane == 0 && mx > 0.f) atomicMax(reinterpret_cast<int*>(P.amax), __float_as_int(mx));
  }
}

template <int EPI>
__device__ __forceinline__ void epi_plain(const Params& p, const EpiUnit& P, const EpiWarp& e,
                                          uint32_t tb, int col0, int cb, int ce) {
#pragma unroll 1
  for (int c = cb; c < ce; c += 32) {
    const int col = col0 + c;
    if (col >= P.N) break;
    uint32_t d[32];
    __syncwarp();
    tmem_ld32(tb + c, d);
    tmem_wait_ld();
    staging_acquire(e);
    if constexpr (EPI == EPI_STORE_BF16_F8) {
      const float deq = P.mult * P.deq;
      uint32_t q[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        q[j] = pack_bf16x2(deq * __uint_as_float(d[2 * j]), deq * __uint_as_float(d[2 * j + 1]));
      stage_bf16(e.stg, e.lane, q);
      flush_chunk<1, 2048, false>(p, P, e, col);
    } else if constexpr (EPI == EPI_STORE_BF16) {
      uint32_t q[16];
      if (P.in0) {
        // the block's residual add: D = alpha * residual + acc
        const __nv_bfloat16* res = static_cast<const __nv_bfloat16*>(P.in0);
        const int row = e.row0 + e.lane;
        const size_t off = static_cast<size_t>(row) * P.ld + col;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 r = (row < P.M && col + 8 * v < P.N) ? ld_global_v4(res + off + 8 * v)
                                                          : make_uint4(0, 0, 0, 0);
          const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = unpack_bf16x2(rw[j]);
            q[4 * v + j] = pack_bf16x2(P.alpha * f.x + __uint_as_float(d[8 * v + 2 * j]),
                                       P.alpha * f.y + __uint_as_float(d[8 * v + 2 * j + 1]));
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          q[j] = pack_bf16x2(__uint_as_float(d[2 * j]), __uint_as_float(d[2 * j + 1]));
      }
      stage_bf16(e.stg, e.lane, q);
      flush_chunk<1, 2048, false>(p, P, e, col);
    } else {
      stage_f32(e.stg, e.lane, d);
      flush_chunk<1, 4096, true>(p, P, e, col);
    }
  }
}

// EPI_FWD_FUSED: the producer thread of a down unit waits (bounded) until
// every gate/up tile of its 256-row block is stored, then orders its TMA
// loads of the postact after that.  False on expiry or abort.
__device__ __forceinline__ bool wait_block_ready(const Params& p, int tm, uint64_t limit_ns,
                                                 volatile int* abort) {
  const int* ctr = p.dep + tm;
  if (ld_acquire_gpu(ctr) < p.dep_target) {
    const uint64_t t0 = globaltimer_ns();
    uint32_t n = 0;
    while (ld_acquire_gpu(ctr) < p.dep_target) {
      if ((++n & 15u) == 0 && (*abort || globaltimer_ns() - t0 > limit_ns)) return false;
      __nanosleep(64);
    }
  }
  fence_proxy_async_global();
  return true;
}

// EPI_FWD_FUSED: one epilogue warp's share of a gate/up tile is stored.  Lane
// 0, which issued the warp's TMA stores, waits for them to complete and
// counts the warp for the tile's 256-row block (release).
__device__ __forceinline__ void signal_block_part(const Params& p, int tm, int lane) {
  if (lane == 0) {
    bulk_wait_all();
    fence_proxy_async_global();
    red_release_gpu_add(p.dep + tm, 1);
  }
  __syncwarp();
}

// -------------------------------------------------------------------- kernel
// Per-CTA-group constants.  CG = 1: one CTA computes a 128 x 256 tile and
// stages all 256 B rows.  CG = 2: a CTA pair computes a 256 x 256 tile with
// one tcgen05.mma.cta_group::2; each CTA stages its own 128 A rows and 128
// of the 256 B rows, so a stage is 32 KB and six fit in shared memory.
// After the stage ring come the epilogue warps' staging buffers; the ring
// takes as many stages as fit beside them in the 227 KB of shared memory.
template <int EPI, int CG>
struct Cfg {
  static constexpr int B_ROWS = CG == 2 ? 128 : 256;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STG = NUM_EPI_WARPS * EpiTraits<EPI>::STG_WARP;
  static constexpr int MAX_SMEM = 232448;  // per-block opt-in limit
  static constexpr int FIT = (MAX_SMEM - 2048 - STG) / STAGE;
  static constexpr int STAGES = FIT < 8 ? FIT : 8;
  static constexpr int TILE_M = BM * CG;
  static constexpr int SMEM = STAGES * STAGE + STG + 1024 /*align*/ + 1024 /*barriers, ring*/;
  static_assert(STAGES >= 2, "stage ring too small");
  static_assert(SMEM <= MAX_SMEM, "shared memory over the limit");
};

// What the producer needs of a work unit, read from the launch parameters
// once per unit and then kept in registers: the TMA issue loop must not go
// back to parameter memory (a generic load, re-issued after every copy's
// memory clobber) for every k-block.
struct UnitLoads {
  const CUtensorMap* a0;  // A operand of segment 0 / 1
  const CUtensorMap* a1;
  const CUtensorMap* b0;  // B operand of segment 0 / 1 (gated: this CTA's gate or up rows)
  const CUtensorMap* b1;
  int m0;                 // this CTA's first A row (K-major) / column (MN-major)
  int n0;                 // this CTA's first B row
  int kb0;                // k-blocks of segment 0
  // derivative epilogues: the saved inputs' tile (this CTA's rows), prefetched into L2
  const CUtensorMap* i0;  // nullptr: none
  const CUtensorMap* i1;
  int icol;               // the tile's first column
  int l2a, l2b;           // the operands' L2 policies (Prob::l2a, l2b)
};

template <int EPI, int CG>
__device__ __forceinline__ UnitLoads unit_loads(const Params& p, const Prob& P, const Work& w,
                                                uint32_t rank) {
  UnitLoads L;
  L.a0 = &p.maps[P.mapA0];
  L.a1 = &p.maps[P.mapA1];
  L.m0 = w.tm * (BM * CG) + static_cast<int>(rank) * BM;
  L.kb0 = P.kb0;
  L.l2a = P.l2a;
  L.l2b = P.l2b;
  if (gated_unit<EPI>(w.prob)) {
    // CG=1: both weights' rows; CG=2: the leader stages the gate rows, the peer the up rows
    L.b0 = &p.maps[(CG == 2 && rank != 0) ? P.mapB1 : P.mapB0];
    L.b1 = &p.maps[P.mapB1];
    L.n0 = w.tn * 128;
  } else {
    L.b0 = &p.maps[P.mapB0];
    L.b1 = &p.maps[P.mapB1];
    L.n0 = w.tn * MMA_N + static_cast<int>(rank) * (MMA_N / CG);
  }
  L.i0 = nullptr;
  L.i1 = nullptr;
  L.icol = w.tn * MMA_N;
  if constexpr (EpiTraits<EPI>::DACT) {
    if (L.m0 < P.M) {  // rows past the output have no inputs to fetch
      if (P.mapI0 >= 0) L.i0 = &p.maps[P.mapI0];
      if (P.mapI1 >= 0) L.i1 = &p.maps[P.mapI1];
    }
  }
  return L;
}

// Issues the TMA boxes of one k-block into this CTA's stage (A at sA, B at
// sB), completing on barrier `full` (for a pair: the leader's barrier).
//   A K-major: one box {64 k, 128 rows};  A MN-major: two boxes {64 m, 64 k}.
//   B gated:   CG=1 the gate and the up rows (two {64, 128} boxes);
//              CG=2 the leader stages the gate rows, the peer the up rows.
//   B K-major: one box {64, 256 / CG};      B MN-major: 4 / CG boxes {64 n, 64 k}.
//   8-bit operands: K-major boxes as above ({128 k, rows}); A MN-major one box
//   {128 m, 128 k}; B MN-major 2 / CG boxes {128 n, 128 k}.
//   EPI_DACT_RECOMP, EPI_DGRAD_F8_RECOMP: segment 0 B K-major (W1), segment 1
//   B MN-major (Wd, W2_8).
template <int EPI, bool A_MN, bool B_MN, int CG>
__device__ __forceinline__ void load_stage(const UnitLoads& L, int seg, int kc, uint32_t sA,
                                           uint32_t sB, uint32_t full, uint64_t polA,
                                           uint64_t polB) {
  uint64_t pol = polA;
  auto ld = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1) {
    if constexpr (CG == 2) tma_load_2d_pair(dst, m, c0, c1, full, pol);
    else tma_load_2d(dst, m, c0, c1, full, pol);
  };
  const CUtensorMap* mA = seg == 0 ? L.a0 : L.a1;
  if constexpr (!A_MN) {
    ld(sA, mA, kc, L.m0);
  } else if constexpr (is_f8(EPI)) {
    ld(sA, mA, L.m0, kc);
  } else {
    ld(sA, mA, L.m0, kc);
    ld(sA + 8192, mA, L.m0 + 64, kc);
  }
  pol = polB;
  if constexpr (EPI == EPI_GATED_FWD) {
    ld(sB, L.b0, kc, L.n0);
    if constexpr (CG == 1) ld(sB + 16384, L.b1, kc, L.n0);
  } else {
    const CUtensorMap* mB = seg == 0 ? L.b0 : L.b1;
    // the fused recomputes read W1 (K-major) in segment 0, Wd (MN-major) in 1
    const bool b_mn = is_recomp(EPI) ? seg == 1 : B_MN;
    if (!b_mn) {
      ld(sB, mB, kc, L.n0);
    } else if constexpr (is_f8(EPI)) {
#pragma unroll
      for (int j = 0; j < 2 / CG; ++j) ld(sB + j * 16384, mB, L.n0 + j * 128, kc);
    } else {
#pragma unroll
      for (int j = 0; j < 4 / CG; ++j) ld(sB + j * 8192, mB, L.n0 + j * 64, kc);
    }
  }
}

// ACT: the activation of the activation epilogues (Act; 0 for the others).
template <int EPI, bool A_MN, bool B_MN, int CG, int ACT>
__global__ void __launch_bounds__(NUM_THREADS, 1) k_mlp_gemm(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  using C = Cfg<EPI, CG>;
  constexpr bool PAIR = CG == 2;
  static_assert(EPI != EPI_FWD_FUSED || CG == 2, "the fused forward runs on CTA pairs");
  // 8-bit operands: a 128-byte k-block row holds 128 elements (bf16: 64)
  constexpr bool F8 = is_f8(EPI);
  constexpr int KE = F8 ? 2 * BK : BK;
  constexpr uint32_t IDESC = idesc_bf16(C::TILE_M, MMA_N, A_MN, B_MN);
  constexpr uint32_t IDESC_BMN = idesc_bf16(C::TILE_M, MMA_N, A_MN, true);

  // 1024-byte aligned stage ring (the 128-byte swizzle repeats every 1 KB)
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* base_g = smem_raw + (base_s - raw_s);
  const uint32_t stg_s = base_s + C::STAGES * C::STAGE;  // epilogue staging
  uint8_t* ctrl = base_g + C::STAGES * C::STAGE + C::STG;
  uint64_t* bar = reinterpret_cast<uint64_t*>(ctrl);
  // barrier indices (same offsets in both CTAs of a pair)
  constexpr int FULL = 0, EMPTY = C::STAGES, TFULL = 2 * C::STAGES, TEMPTY = 2 * C::STAGES + 2,
                SFULL = 2 * C::STAGES + 4, SEMPTY = 2 * C::STAGES + 4 + SCHED_SLOTS,
                DRAIN = 2 * C::STAGES + 4 + 2 * SCHED_SLOTS;
  // EPI_DGRAD_F8: two barriers per epilogue warp for its TMA-loaded preact boxes
  constexpr int EBAR = DRAIN + 1;
  constexpr int NBAR = EBAR + 2 * NUM_EPI_WARPS;
  int* sched = reinterpret_cast<int*>(ctrl + 8 * NBAR);
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(sched + SCHED_SLOTS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_s + 1);
  auto bar_s = [&](int i) { return smem_u32(bar + i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  // the leader's copy of a barrier / ring slot, as a shared::cluster address
  auto lead = [&](uint32_t local) { return PAIR ? mapa_shared(local, 0) : local; };
  auto peer = [&](uint32_t local) { return mapa_shared(local, 1); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(bar_s(FULL + i), 1);
      mbar_init(bar_s(EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s(TFULL + i), 1);
      mbar_init(bar_s(TEMPTY + i), CG * NUM_EPI_WARPS);
    }
    for (int i = 0; i < SCHED_SLOTS; ++i) {
      mbar_init(bar_s(SFULL + i), 1);
      // MMA issuer + every epilogue warp of the pair + the peer's producer
      mbar_init(bar_s(SEMPTY + i), 1 + CG * NUM_EPI_WARPS + (CG - 1));
    }
    mbar_init(bar_s(DRAIN), 1);
    if constexpr (EPI == EPI_DGRAD_F8)
      for (int i = 0; i < 2 * NUM_EPI_WARPS; ++i) mbar_init(bar_s(EBAR + i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Work units come from the atomic counter.  A cluster's first unit is its
  // cluster id, so it starts without the atomic's round trip and a launch of
  // about one unit per cluster gets one unit to each cluster however late
  // some start; the units of such launches do not depend on one another.
  // The fused forward's down units wait for gate/up tiles, so there every
  // unit, the first included, is claimed from the counter: a cluster that is
  // not resident yet owns no unit, and a down unit only ever waits for
  // gate/up tiles that running clusters have claimed.  (The counter was
  // cleared before the call's first kernel started, so this claim need not
  // wait for the previous kernel.)
  constexpr bool CLAIM_ALL = EPI == EPI_FWD_FUSED;
  int first_unit = static_cast<int>(blockIdx.x) / CG;
  if (warp == 0 && lane == 0) {
    if (CLAIM_ALL && leader) first_unit = atomicAdd(p.counter, 1);
    for (int i = 0; i < p.nmaps; ++i) prefetch_tmap(&p.maps[i]);
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(tmem_base_s), TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync();  // barriers of both CTAs initialised before remote use
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;

  // Inputs written by the previous kernel on the stream are visible after this.
  pdl_wait();
  pdl_launch_dependents();

  const uint64_t lim = p.timeout_ns;
  const int ncl = gridDim.x / CG;          // clusters (CTA groups) in the grid

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_n = policy_evict_normal(), pol_l = policy_evict_last(),
                     pol_f = policy_evict_first();
      auto pol_of = [&](int k) { return k == 1 ? pol_l : (k == 2 ? pol_f : pol_n); };
      const uint32_t tx_bytes = CG * (p.a_tx_bytes + C::B_BYTES);
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t sphase = 0;
      int issued = 0;  // k-blocks issued (for the drain on abort)
      int unit = first_unit;
      bool ok = true;
      // testing hook: publish no work, so the consumers' bounded waits expire
      const bool publish_nothing = leader && (p.debug_flags & 1);
      bool first_pub = true;
      while (ok && !publish_nothing) {
        if (leader) {
          // Publishes unit v (-1: no more work) to the pair's rings.  A unit
          // is published while the previous one is still being loaded (at
          // its middle k-block), so that the peer and the consumers find it
          // in the ring when they get there.  Kernels with an MN-major A
          // (the weight gradients) publish each unit as they start loading
          // it instead: measured, the early publication made them 1-3 %
          // slower while it made the others 1-7 % faster.
          auto publish = [&](int v) -> bool {
            if (!mbar_wait<PAIR>(bar_s(SEMPTY + slot), sphase ^ 1u, lim, abort_flag)) return false;
            sched[slot] = v;
            if constexpr (PAIR) {
              st_shared_cluster_u32(peer(smem_u32(sched + slot)), static_cast<uint32_t>(v));
              mbar_arrive_cluster(peer(bar_s(SFULL + slot)));
            }
            mbar_arrive(bar_s(SFULL + slot));
            if (++slot == SCHED_SLOTS) { slot = 0; sphase ^= 1u; }
            return true;
          };
          constexpr bool EARLY_PUB = !A_MN;
          if (!EARLY_PUB || first_pub) {
            first_pub = false;
            if (!publish(unit < p.total_units ? unit : -1)) {
              ok = false;
              break;
            }
          }
          if (unit >= p.total_units) break;
          const Work w = decode_unit(p, unit);
          // The next unit, fetched now and needed when it is published.  A
          // down unit of the fused forward (K = I, several times a gate/up
          // unit's length) fetches it only when it publishes it, half-way
          // through: fetched at its start, the last down units of the queue
          // went two to a pair while other pairs found the queue empty, and
          // a forward of a few hundred tokens took one down unit longer.
          const bool late_claim = CLAIM_ALL && w.prob == 1;
          int next = late_claim ? -1 : (CLAIM_ALL ? 0 : ncl) + atomicAdd(p.counter, 1);
          auto claim = [&] {
            if (late_claim) next = atomicAdd(p.counter, 1);
          };
          bool published = !EARLY_PUB;
          const UnitLoads L = unit_loads<EPI, CG>(p, p.prob[w.prob], w, rank);
          if constexpr (EpiTraits<EPI>::DACT) {
            // the epilogue reads this tile's saved inputs a tile or two later
            if (L.i0) tma_prefetch_l2_2d(L.i0, L.icol, L.m0);
            if (L.i1) tma_prefetch_l2_2d(L.i1, L.icol, L.m0);
          }
          if constexpr (EPI == EPI_FWD_FUSED) {
            // a down unit reads the postact of its rows
            if (w.prob == 1 && !wait_block_ready(p, w.tm, lim, abort_flag)) {
              ok = false;
              break;
            }
          }
          for (int kb = w.kb_begin; kb < w.kb_end && ok; ++kb) {
            if (!mbar_wait<PAIR>(bar_s(EMPTY + stage), phase ^ 1u, lim, abort_flag)) {
              ok = false;
              break;
            }
            const uint32_t full = bar_s(FULL + stage);
            // the leader's full barrier expects the bytes of both CTAs of a pair
            // (the A boxes of an output with few rows cover only those rows)
            mbar_expect_tx(full, tx_bytes);
            const int seg = kb < L.kb0 ? 0 : 1;
            const int kc = (seg == 0 ? kb : kb - L.kb0) * KE;
            const uint32_t sA = base_s + stage * C::STAGE;
            load_stage<EPI, A_MN, B_MN, CG>(L, seg, kc, sA, sA + C::A_BYTES, full,
                                            pol_of(L.l2a), pol_of(L.l2b));
            ++issued;
            if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
            if (!published && kb == w.kb_begin + (w.kb_end - w.kb_begin) / 2) {
              claim();
              if (!publish(next < p.total_units ? next : -1)) {
                ok = false;
                break;
              }
              published = true;
            }
          }
          if (ok && !published) {
            claim();
            if (!publish(next < p.total_units ? next : -1)) ok = false;
          }
          unit = next;
        } else {
          // peer of a pair: take units from the ring the leader fills
          if (!mbar_wait<PAIR>(bar_s(SFULL + slot), sphase, lim, abort_flag)) {
            ok = false;
            break;
          }
          const int v = sched[slot];
          mbar_arrive_cluster(lead(bar_s(SEMPTY + slot)));
          if (++slot == SCHED_SLOTS) { slot = 0; sphase ^= 1u; }
          if (v < 0) break;
          const Work w = decode_unit(p, v);
          const UnitLoads L = unit_loads<EPI, CG>(p, p.prob[w.prob], w, rank);
          if constexpr (EpiTraits<EPI>::DACT) {
            if (L.i0) tma_prefetch_l2_2d(L.i0, L.icol, L.m0);
            if (L.i1) tma_prefetch_l2_2d(L.i1, L.icol, L.m0);
          }
          if constexpr (EPI == EPI_FWD_FUSED) {
            if (w.prob == 1 && !wait_block_ready(p, w.tm, lim, abort_flag)) {
              ok = false;
              break;
            }
          }
          const uint32_t full_lead = lead(bar_s(FULL));
          for (int kb = w.kb_begin; kb < w.kb_end && ok; ++kb) {
            if (!mbar_wait<PAIR>(bar_s(EMPTY + stage), phase ^ 1u, lim, abort_flag)) {
              ok = false;
              break;
            }
            const int seg = kb < L.kb0 ? 0 : 1;
            const int kc = (seg == 0 ? kb : kb - L.kb0) * KE;
            const uint32_t sA = base_s + stage * C::STAGE;
            load_stage<EPI, A_MN, B_MN, CG>(L, seg, kc, sA, sA + C::A_BYTES,
                                            full_lead + 8u * stage, pol_of(L.l2a),
                                            pol_of(L.l2b));
            ++issued;
            if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
      if (!ok) {
        record_timeout(p, abort_flag);
        if (leader) {
          // let the copies already in flight land before shared memory is released
          int s = stage;
          uint32_t ph = phase;
          for (int i = 0; i < C::STAGES && i < issued; ++i) {
            if (--s < 0) { s = C::STAGES - 1; ph ^= 1u; }
            volatile int never = 0;
            mbar_wait<PAIR>(bar_s(FULL + s), ph, 10000000ull, &never);
          }
        } else {
          __nanosleep(100000);  // the peer's copies signal the leader's barriers
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      // 8-bit operands: their formats come with the launch
      // (the 8-bit fused recompute: segment 0's formats and K-major B, then
      // segment 1's with B MN-major)
      const uint32_t idesc_8 = idesc_f8(C::TILE_M, MMA_N, p.f8_formats & 7, (p.f8_formats >> 3) & 7,
                                        A_MN, B_MN || is_recomp(EPI));
      const uint32_t idesc_8s0 = idesc_f8(C::TILE_M, MMA_N, p.f8_formats0 & 7,
                                          (p.f8_formats0 >> 3) & 7, A_MN, false);
      (void)idesc_8;
      (void)idesc_8s0;
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t sphase = 0;
      int acc = 0;
      uint32_t aphase = 0;
      bool ok = true;
      bool any = false;
      while (ok) {
        if (!mbar_wait<PAIR>(bar_s(SFULL + slot), sphase, lim, abort_flag)) { ok = false; break; }
        const int unit = sched[slot];
        mbar_arrive(bar_s(SEMPTY + slot));
        if (++slot == SCHED_SLOTS) { slot = 0; sphase ^= 1u; }
        if (unit < 0) break;
        const Work w = decode_unit(p, unit);
        // the fused recompute's second K segment goes to the other accumulator
        const int kswitch = is_recomp(EPI) ? p.prob[w.prob].kb0 : -1;
        if (!mbar_wait<PAIR>(bar_s(TEMPTY + acc), aphase ^ 1u, lim, abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint32_t d = tmem + acc * MMA_N;
        int kfirst = w.kb_begin;
        bool seg1 = false;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (is_recomp(EPI) && kb == kswitch) {
            if constexpr (PAIR) tc_commit_pair(bar_s(TFULL + acc), 3);
            else tc_commit(bar_s(TFULL + acc));
            acc ^= 1;
            if (acc == 0) aphase ^= 1u;
            if (!mbar_wait<PAIR>(bar_s(TEMPTY + acc), aphase ^ 1u, lim, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d = tmem + acc * MMA_N;
            kfirst = kb;
            seg1 = true;
          }
          if (!mbar_wait<PAIR>(bar_s(FULL + stage), phase, lim, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = base_s + stage * C::STAGE;
          const uint32_t sB = sA + C::A_BYTES;
          const bool b_mn = B_MN || seg1;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // MN-major: bf16 K=16 steps of 16 rows, 8-bit K=32 steps of 32 rows
            constexpr uint32_t MN_STEP = F8 ? 4096 : 2048, MN_LBO = F8 ? 16384 : 8192;
            const uint64_t ad = A_MN ? sdesc_sw128(sA + k * MN_STEP, MN_LBO, 1024)
                                     : sdesc_sw128(sA + k * 32, 16, 1024);
            const uint64_t bd = b_mn ? sdesc_sw128(sB + k * MN_STEP, MN_LBO, 1024)
                                     : sdesc_sw128(sB + k * 32, 16, 1024);
            const uint32_t idesc =
                F8 ? ((is_recomp(EPI) && !seg1) ? idesc_8s0 : idesc_8) : b_mn ? IDESC_BMN : IDESC;
            const uint32_t accum = (kb > kfirst || k > 0) ? 1u : 0u;
            if constexpr (F8) {
              if constexpr (PAIR) tc_mma_f8_pair(d, ad, bd, idesc, accum);
              else tc_mma_f8(d, ad, bd, idesc, accum);
            } else {
              if constexpr (PAIR) tc_mma_bf16_pair(d, ad, bd, idesc, accum);
              else tc_mma_bf16(d, ad, bd, idesc, accum);
            }
          }
          any = true;
          if constexpr (PAIR) tc_commit_pair(bar_s(EMPTY + stage), 3);
          else tc_commit(bar_s(EMPTY + stage));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if constexpr (PAIR) tc_commit_pair(bar_s(TFULL + acc), 3);
        else tc_commit(bar_s(TFULL + acc));
        acc ^= 1;
        if (acc == 0) aphase ^= 1u;
      }
      if (!ok) {
        record_timeout(p, abort_flag);
        if (any) {  // wait for the MMAs already issued before TMEM is freed
          if constexpr (PAIR) tc_commit_pair(bar_s(DRAIN), 1);
          else tc_commit(bar_s(DRAIN));
          volatile int never = 0;
          mbar_wait<PAIR>(bar_s(DRAIN), 0, 10000000ull, &never);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;  // which half of the tile's columns
    EpiWarp e;
    e.stg = stg_s + static_cast<uint32_t>(warp - 2) * EpiTraits<EPI>::STG_WARP;
    e.lane = lane;
    e.box = 0;
    e.ebar = bar_s(EBAR + 2 * (warp - 2));
    e.ephase = 0;
    e.epend = 0;
    const uint64_t epol = policy_evict_normal();  // the epilogue's TMA loads
    int slot = 0;
    uint32_t sphase = 0;
    int acc = 0;
    uint32_t aphase = 0;
    // 8-bit epilogues: each problem's dequant factor *sa * *sb and output
    // quantisation factor 1 / *sq (device scalars), read once
    float f8_deq[MAX_PROBS], f8_inv[MAX_PROBS];
    float f8_deq0 = 1.f;  // EPI_DGRAD_F8_RECOMP (one problem): the recomputed preact's
#pragma unroll
    for (int i = 0; i < MAX_PROBS; ++i) {
      f8_deq[i] = 1.f;
      f8_inv[i] = 1.f;
      if constexpr (is_f8(EPI)) {
        if (i < p.nprob) {
          f8_deq[i] = *p.prob[i].sa * *p.prob[i].sb;
          if (p.prob[i].sq) f8_inv[i] = 1.0f / *p.prob[i].sq;
        }
      }
    }
    if constexpr (EPI == EPI_DGRAD_F8_RECOMP) f8_deq0 = *p.prob[0].sp0 * *p.prob[0].sp1;
    while (true) {
      if (!mbar_wait<PAIR>(bar_s(SFULL + slot), sphase, lim, abort_flag)) {
        record_timeout(p, abort_flag);
        break;
      }
      const int unit = sched[slot];
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(bar_s(SEMPTY + slot));
        else mbar_arrive_cluster(lead(bar_s(SEMPTY + slot)));
      }
      if (++slot == SCHED_SLOTS) { slot = 0; sphase ^= 1u; }
      if (unit < 0) break;
      const Work w = decode_unit(p, unit);
      const int pi = w.prob;
      const EpiUnit P = epi_unit<EPI>(p, p.prob[pi],
                                      pi == 0 ? f8_deq[0] : pi == 1 ? f8_deq[1] : f8_deq[2],
                                      pi == 0 ? f8_inv[0] : pi == 1 ? f8_inv[1] : f8_inv[2],
                                      f8_deq0);
      e.row0 = w.tm * C::TILE_M + static_cast<int>(rank) * BM + q * 32;
      e.rows_ok = e.row0 < P.M;
      e.rs = (P.rstd && e.row0 + lane < P.M) ? P.rstd[e.row0 + lane] : 1.f;
      const int tile_n = tile_n_of<EPI>(pi);
      const int cb = half * (tile_n / 2), ce = cb + tile_n / 2;
      const int col0 = w.tn * tile_n;
      uint4 pg[4], pu[4];
      // s*act'(p) (bf16: dd = 2 relu(pre)) between the two phases
      uint32_t dd[is_recomp(EPI) ? 64 : 1];
      (void)dd;
      if constexpr (is_recomp(EPI)) {
        // phase 1 on the recomputed preact, then its accumulator goes back to the MMAs
        if (!mbar_wait<PAIR>(bar_s(TFULL + acc), aphase, lim, abort_flag)) {
          record_timeout(p, abort_flag);
          break;
        }
        tc_fence_after();
        if (e.rows_ok) {
          const uint32_t t0 = tmem + acc * MMA_N + (static_cast<uint32_t>(q * 32) << 16);
          if constexpr (EPI == EPI_DACT_RECOMP) epi_recomp_p<ACT>(p, P, e, t0, col0, cb, dd);
          else epi_recomp_f8_p(P, t0, col0, cb, dd);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(bar_s(TEMPTY + acc));
          else mbar_arrive_cluster(lead(bar_s(TEMPTY + acc)));
        }
        acc ^= 1;
        if (acc == 0) aphase ^= 1u;
      }
      if constexpr (EpiTraits<EPI>::DACT) {
        // the saved preacts do not depend on the MMAs: fetch the first chunk(s) now
        if (EPI == EPI_DGRAD_F8 && P.ein != nullptr) {
          if (e.rows_ok) {
            staging_acquire(e);  // the previous tile's store has read the box
            dgrad_f8_issue(P, e, col0 + cb, 0, epol);
            dgrad_f8_issue(P, e, col0 + cb + 32, 1, epol);
          }
        } else if (e.rows_ok) {
          dact_load_rows<EPI == EPI_DGATED>(P, e.row0, lane, col0 + cb, pg, pu);
        }
      }
      if (!mbar_wait<PAIR>(bar_s(TFULL + acc), aphase, lim, abort_flag)) {
        record_timeout(p, abort_flag);
        if constexpr (EPI == EPI_DGRAD_F8) dgrad_f8_drain(e);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + acc * MMA_N + (static_cast<uint32_t>(q * 32) << 16);
      if (e.rows_ok) {  // warp-uniform: rows past the output need no epilogue
        if constexpr (EPI == EPI_GATED_FWD) {
          epi_gated_fwd<ACT>(p, P, e, tb, col0, cb, ce);
        } else if constexpr (EPI == EPI_FWD_FUSED) {
          if (pi == 0) epi_gated_fwd<ACT>(p, P, e, tb, col0, cb, ce);
          else epi_plain<EPI_STORE_BF16>(p, P, e, tb, col0, cb, ce);
        } else if constexpr (EPI == EPI_ACT_FWD) {
          epi_act_fwd<ACT>(p, P, e, tb, col0, cb, ce);
        } else if constexpr (EPI == EPI_DGATED) {
          epi_dact<ACT, true>(p, P, e, tb, col0, cb, ce, pg, pu);
        } else if constexpr (EPI == EPI_DACT) {
          epi_dact<ACT, false>(p, P, e, tb, col0, cb, ce, pg, pu);
        } else if constexpr (EPI == EPI_DACT_RECOMP) {
          epi_recomp_dh(p, P, e, tb, col0, cb, dd);
        } else if constexpr (EPI == EPI_ACT_FWD_F8) {
          epi_act_f8<ACT>(p, P, e, tb, col0, cb, ce);
        } else if constexpr (EPI == EPI_DGRAD_F8) {
          if (P.ein == nullptr) {
            epi_dgrad_f8(p, P, e, tb, col0, cb, ce, pg);
          } else if (!epi_dgrad_f8_tma(P, e, tb, col0, cb, lim, abort_flag, epol)) {
            record_timeout(p, abort_flag);
            break;
          }
        } else if constexpr (EPI == EPI_DGRAD_F8_RECOMP) {
          epi_recomp_f8_dh(P, e, tb, col0, cb, dd);
        } else {
          epi_plain<EPI>(p, P, e, tb, col0, cb, ce);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(bar_s(TEMPTY + acc));
        else mbar_arrive_cluster(lead(bar_s(TEMPTY + acc)));
      }
      acc ^= 1;
      if (acc == 0) aphase ^= 1u;
      if constexpr (EPI == EPI_FWD_FUSED) {
        // the down units of this block wait for every warp's gate/up stores
        if (pi == 0) signal_block_part(p, w.tm, lane);
      }
    }
    // the last stores must finish before the kernel (and its shared memory) ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  if constexpr (PAIR) cluster_sync();  // no remote arrival or copy may target an exited CTA
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem, TMEM_COLS);
  }
}

template <int EPI, bool A_MN, bool B_MN, int CG, int ACT>
cudaError_t launch_gemm(const Params& p, int grid, cudaStream_t stream, bool pdl) {
  auto kern = k_mlp_gemm<EPI, A_MN, B_MN, CG, ACT>;
  static std::atomic<unsigned> configured_dev_mask{0};  // devices that got the smem attribute
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 31 || !(configured_dev_mask.load() & (1u << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<EPI, CG>::SMEM);
    if (e != cudaSuccess) return e;
    if (CG == 2) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
      (void)e;
    }
    if (dev < 31) configured_dev_mask.fetch_or(1u << dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<EPI, CG>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (CG == 2) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Largest number of CTA pairs that can be co-resident (0 on error).
template <int EPI, bool A_MN, bool B_MN, int CG, int ACT>
int max_groups() {
  auto kern = k_mlp_gemm<EPI, A_MN, B_MN, CG, ACT>;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (CG == 1) return sms;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<EPI, CG>::SMEM) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<EPI, CG>::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
  return n;
}

}  // namespace mlpk
