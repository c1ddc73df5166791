// gemm.cuh -- the persistent, warp-specialised tcgen05 GEMM with the MLP's
// fused epilogues.
//
// One CTA per SM (192 threads, ~195 KB shared memory, all 512 TMEM columns):
//   warp 0     TMA producer and tile scheduler: fetches work units from a
//              global atomic counter (first unit = blockIdx.x), publishes
//              them through a shared-memory ring, and streams the A/B
//              k-blocks of each unit into a 4-stage shared-memory ring.
//   warp 1     allocates TMEM; one lane issues tcgen05.mma (M=128, N=256,
//              K=16) into one of two 256-column fp32 accumulators and
//              commits stage releases / accumulator-full signals.
//   warps 2-5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//              32*(w%4)..+31, i.e. one output row per thread), apply the
//              fused activation / derivative / scaling, store to global.
// The double-buffered accumulator lets the epilogue of tile t overlap the
// MMAs of tile t+1.  Every wait is bounded (globaltimer); on expiry the
// kernel records MLP_ERR_TIMEOUT in the status word and unwinds.
//
// Operand layouts.  A is BM x BK, B is 256 x BK, both bf16 with the
// 128-byte swizzle.  K-major operands ([rows, K], K contiguous) arrive as
// one TMA box {64 (K), rows}; MN-major operands ([K, MN], MN contiguous)
// arrive as boxes {64 (MN), 64 (K)} placed 8 KB apart.  The matching UMMA
// descriptors: K-major SBO = 1024 B (8-row groups), start += 32 B per K=16
// step; MN-major LBO = 8192 B (next 64-wide MN block), SBO = 1024 B (next 8
// K rows), start += 2048 B per K=16 step.
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
  int per_group = p.group_m * P.tiles_n;
  int g = t / per_group;
  int first_m = g * p.group_m;
  int gsz = min(P.tiles_m - first_m, p.group_m);
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

template <int EPI>
struct EpiTraits {
  static constexpr int TILE_N = (EPI == EPI_GATED_FWD) ? 128 : 256;
};

__device__ __forceinline__ void record_timeout(const Params& p, volatile int* abort_flag) {
  *abort_flag = 1;
  if (p.status) atomicExch(p.status, MLP_ERR_TIMEOUT_CODE);
}

// ---------------------------------------------------------------- epilogues
// Each thread owns one output row `row` of the tile and walks its columns in
// chunks of 32 (one tcgen05.ld 32x32b.x32).  tcgen05.ld is warp-collective,
// so every lane issues it whatever its row's validity.

template <int ACT>
__device__ __forceinline__ void epi_gated_fwd(const Params& p, const Prob& P, uint32_t tb, int row,
                                              int col0) {
  const bool row_ok = row < P.M;
  const float s = p.scale;
  __nv_bfloat16* a_out = static_cast<__nv_bfloat16*>(P.out0);
  __nv_bfloat16* g_out = static_cast<__nv_bfloat16*>(P.out1);
  __nv_bfloat16* u_out = static_cast<__nv_bfloat16*>(P.out2);
#pragma unroll 1
  for (int c = 0; c < 128; c += 32) {
    uint32_t g[32], u[32];
    __syncwarp();
    tmem_ld32(tb + c, g);
    tmem_ld32(tb + 128 + c, u);
    tmem_wait_ld();
    const int col = col0 + c;
    if (row_ok && col < P.N) {
      const size_t off = static_cast<size_t>(row) * P.ld + col;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        if (col + 8 * v < P.N) {
          uint32_t pa[4], pg[4], pu[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float g0 = __uint_as_float(g[8 * v + 2 * j]), g1 = __uint_as_float(g[8 * v + 2 * j + 1]);
            float u0 = __uint_as_float(u[8 * v + 2 * j]), u1 = __uint_as_float(u[8 * v + 2 * j + 1]);
            pa[j] = pack_bf16x2(s * act_f<ACT>(g0) * u0, s * act_f<ACT>(g1) * u1);
            pg[j] = pack_bf16x2(g0, g1);
            pu[j] = pack_bf16x2(u0, u1);
          }
          if (a_out) st_global_v4(a_out + off + 8 * v, make_uint4(pa[0], pa[1], pa[2], pa[3]));
          if (g_out) st_global_v4(g_out + off + 8 * v, make_uint4(pg[0], pg[1], pg[2], pg[3]));
          if (u_out) st_global_v4(u_out + off + 8 * v, make_uint4(pu[0], pu[1], pu[2], pu[3]));
        }
      }
    }
  }
}

template <int ACT>
__device__ __forceinline__ void epi_act_fwd(const Params& p, const Prob& P, uint32_t tb, int row,
                                            int col0) {
  const bool row_ok = row < P.M;
  const float s = p.scale;
  __nv_bfloat16* a_out = static_cast<__nv_bfloat16*>(P.out0);
  __nv_bfloat16* p_out = static_cast<__nv_bfloat16*>(P.out1);
#pragma unroll 1
  for (int c = 0; c < 256; c += 32) {
    uint32_t z[32];
    __syncwarp();
    tmem_ld32(tb + c, z);
    tmem_wait_ld();
    const int col = col0 + c;
    if (row_ok && col < P.N) {
      const size_t off = static_cast<size_t>(row) * P.ld + col;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        if (col + 8 * v < P.N) {
          uint32_t pa[4], pp[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float z0 = __uint_as_float(z[8 * v + 2 * j]), z1 = __uint_as_float(z[8 * v + 2 * j + 1]);
            pa[j] = pack_bf16x2(s * act_f<ACT>(z0), s * act_f<ACT>(z1));
            pp[j] = pack_bf16x2(z0, z1);
          }
          if (a_out) st_global_v4(a_out + off + 8 * v, make_uint4(pa[0], pa[1], pa[2], pa[3]));
          if (p_out) st_global_v4(p_out + off + 8 * v, make_uint4(pp[0], pp[1], pp[2], pp[3]));
        }
      }
    }
  }
}

// GATED = true: in0 = G, in1 = U -> out0 = dG, out1 = dU, out2 = a (optional)
// GATED = false: in0 = P -> out0 = dP, out2 = a (optional)
template <int ACT, bool GATED>
__device__ __forceinline__ void epi_dact(const Params& p, const Prob& P, uint32_t tb, int row,
                                         int col0) {
  const bool row_ok = row < P.M;
  const float s = p.scale;
  const __nv_bfloat16* g_in = static_cast<const __nv_bfloat16*>(P.in0);
  const __nv_bfloat16* u_in = static_cast<const __nv_bfloat16*>(P.in1);
  __nv_bfloat16* dg_out = static_cast<__nv_bfloat16*>(P.out0);
  __nv_bfloat16* du_out = static_cast<__nv_bfloat16*>(P.out1);
  __nv_bfloat16* a_out = static_cast<__nv_bfloat16*>(P.out2);
#pragma unroll 1
  for (int c = 0; c < 256; c += 32) {
    uint32_t d[32];
    __syncwarp();
    tmem_ld32(tb + c, d);
    tmem_wait_ld();
    const int col = col0 + c;
    if (row_ok && col < P.N) {
      const size_t off = static_cast<size_t>(row) * P.ld + col;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        if (col + 8 * v < P.N) {
          uint4 gv = ld_global_v4(g_in + off + 8 * v);
          uint4 uv = GATED ? ld_global_v4(u_in + off + 8 * v) : make_uint4(0, 0, 0, 0);
          const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
          const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
          uint32_t pdg[4], pdu[4], pa[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float2 gg = unpack_bf16x2(gw[j]);
            float dh0 = s * __uint_as_float(d[8 * v + 2 * j]);
            float dh1 = s * __uint_as_float(d[8 * v + 2 * j + 1]);
            float a0, da0, a1, da1;
            act_and_grad<ACT>(gg.x, a0, da0);
            act_and_grad<ACT>(gg.y, a1, da1);
            if (GATED) {
              float2 uu = unpack_bf16x2(uw[j]);
              pdg[j] = pack_bf16x2(dh0 * uu.x * da0, dh1 * uu.y * da1);
              pdu[j] = pack_bf16x2(dh0 * a0, dh1 * a1);
              pa[j] = pack_bf16x2(s * a0 * uu.x, s * a1 * uu.y);
            } else {
              pdg[j] = pack_bf16x2(dh0 * da0, dh1 * da1);
              pa[j] = pack_bf16x2(s * a0, s * a1);
            }
          }
          st_global_v4(dg_out + off + 8 * v, make_uint4(pdg[0], pdg[1], pdg[2], pdg[3]));
          if (GATED) st_global_v4(du_out + off + 8 * v, make_uint4(pdu[0], pdu[1], pdu[2], pdu[3]));
          if (a_out) st_global_v4(a_out + off + 8 * v, make_uint4(pa[0], pa[1], pa[2], pa[3]));
        }
      }
    }
  }
}

template <int EPI>
__device__ __forceinline__ void epi_plain(const Prob& P, uint32_t tb, int row, int col0) {
  const bool row_ok = row < P.M;
#pragma unroll 1
  for (int c = 0; c < 256; c += 32) {
    uint32_t d[32];
    __syncwarp();
    tmem_ld32(tb + c, d);
    tmem_wait_ld();
    const int col = col0 + c;
    if (row_ok && col < P.N) {
      const size_t off = static_cast<size_t>(row) * P.ld + col;
      if constexpr (EPI == EPI_STORE_BF16) {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(P.out0);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          if (col + 8 * v < P.N) {
            uint32_t q[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              q[j] = pack_bf16x2(__uint_as_float(d[8 * v + 2 * j]),
                                 __uint_as_float(d[8 * v + 2 * j + 1]));
            st_global_v4(o + off + 8 * v, make_uint4(q[0], q[1], q[2], q[3]));
          }
        }
      } else {
        float* o = static_cast<float*>(P.out0);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          if (col + 8 * v < P.N) {
            red_add_v4_f32(o + off + 8 * v, __uint_as_float(d[8 * v + 0]),
                           __uint_as_float(d[8 * v + 1]), __uint_as_float(d[8 * v + 2]),
                           __uint_as_float(d[8 * v + 3]));
            red_add_v4_f32(o + off + 8 * v + 4, __uint_as_float(d[8 * v + 4]),
                           __uint_as_float(d[8 * v + 5]), __uint_as_float(d[8 * v + 6]),
                           __uint_as_float(d[8 * v + 7]));
          }
        }
      }
    }
  }
}

// -------------------------------------------------------------------- kernel
template <int EPI, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1) k_mlp_gemm(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int TILE_N = EpiTraits<EPI>::TILE_N;
  constexpr uint32_t IDESC = idesc_bf16(BM, MMA_N, A_MN, B_MN);

  // 1024-byte aligned stage ring (the 128-byte swizzle repeats every 1 KB)
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* base_g = smem_raw + (base_s - raw_s);
  uint8_t* ctrl = base_g + STAGES * STAGE_BYTES;
  uint64_t* bar = reinterpret_cast<uint64_t*>(ctrl);
  // barrier indices
  const int FULL = 0, EMPTY = STAGES, TFULL = 2 * STAGES, TEMPTY = 2 * STAGES + 2,
            SFULL = 2 * STAGES + 4, SEMPTY = 2 * STAGES + 4 + SCHED_SLOTS,
            DRAIN = 2 * STAGES + 4 + 2 * SCHED_SLOTS;
  const int NBAR = DRAIN + 1;
  int* sched = reinterpret_cast<int*>(ctrl + 8 * NBAR);
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(sched + SCHED_SLOTS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_s + 1);
  auto bar_s = [&](int i) { return smem_u32(bar + i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bar_s(FULL + i), 1);
      mbar_init(bar_s(EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s(TFULL + i), 1);
      mbar_init(bar_s(TEMPTY + i), 4);
    }
    for (int i = 0; i < SCHED_SLOTS; ++i) {
      mbar_init(bar_s(SFULL + i), 1);
      mbar_init(bar_s(SEMPTY + i), 5);
    }
    mbar_init(bar_s(DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < MAX_MAPS; ++i) prefetch_tmap(&p.maps[i]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_base_s), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;

  // Inputs written by the previous kernel on the stream are visible after this.
  pdl_wait();
  pdl_launch_dependents();

  const uint64_t lim = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t sphase = 0;
      int issued = 0;  // k-blocks issued (for the drain on abort)
      int unit = blockIdx.x;
      bool ok = true;
      while (ok) {
        const bool done = unit >= p.total_units;
        const int next = done ? unit : (int)gridDim.x + atomicAdd(p.counter, 1);
        if (!mbar_wait(bar_s(SEMPTY + slot), sphase ^ 1u, lim, abort_flag)) {
          ok = false;
          break;
        }
        sched[slot] = done ? -1 : unit;
        mbar_arrive(bar_s(SFULL + slot));
        if (++slot == SCHED_SLOTS) { slot = 0; sphase ^= 1u; }
        if (done) break;
        const Work w = decode_unit(p, unit);
        const Prob& P = p.prob[w.prob];
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!mbar_wait(bar_s(EMPTY + stage), phase ^ 1u, lim, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t full = bar_s(FULL + stage);
          mbar_expect_tx(full, STAGE_BYTES);
          const int seg = kb < P.kb0 ? 0 : 1;
          const int kc = (seg == 0 ? kb : kb - P.kb0) * BK;
          const CUtensorMap* mA = &p.maps[seg == 0 ? P.mapA0 : P.mapA1];
          const uint32_t sA = base_s + stage * STAGE_BYTES;
          const uint32_t sB = sA + A_STAGE_BYTES;
          if constexpr (!A_MN) {
            tma_load_2d(sA, mA, kc, w.tm * BM, full, pol);
          } else {
            tma_load_2d(sA, mA, w.tm * BM, kc, full, pol);
            tma_load_2d(sA + 8192, mA, w.tm * BM + 64, kc, full, pol);
          }
          if constexpr (EPI == EPI_GATED_FWD) {
            tma_load_2d(sB, &p.maps[P.mapB0], kc, w.tn * 128, full, pol);
            tma_load_2d(sB + 16384, &p.maps[P.mapB1], kc, w.tn * 128, full, pol);
          } else {
            const CUtensorMap* mB = &p.maps[seg == 0 ? P.mapB0 : P.mapB1];
            if constexpr (!B_MN) {
              tma_load_2d(sB, mB, kc, w.tn * MMA_N, full, pol);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) tma_load_2d(sB + j * 8192, mB, w.tn * MMA_N + j * 64, kc, full, pol);
            }
          }
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        unit = next;
      }
      if (!ok) {
        record_timeout(p, abort_flag);
        // let the copies already in flight land before shared memory is released
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < STAGES && i < issued; ++i) {
          if (--s < 0) { s = STAGES - 1; ph ^= 1u; }
          volatile int never = 0;
          mbar_wait(bar_s(FULL + s), ph, 10000000ull, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t sphase = 0;
      int acc = 0;
      uint32_t aphase = 0;
      bool ok = true;
      bool any = false;
      while (ok) {
        if (!mbar_wait(bar_s(SFULL + slot), sphase, lim, abort_flag)) { ok = false; break; }
        const int unit = sched[slot];
        mbar_arrive(bar_s(SEMPTY + slot));
        if (++slot == SCHED_SLOTS) { slot = 0; sphase ^= 1u; }
        if (unit < 0) break;
        const Work w = decode_unit(p, unit);
        if (!mbar_wait(bar_s(TEMPTY + acc), aphase ^ 1u, lim, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + acc * MMA_N;
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!mbar_wait(bar_s(FULL + stage), phase, lim, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = base_s + stage * STAGE_BYTES;
          const uint32_t sB = sA + A_STAGE_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = A_MN ? sdesc_sw128(sA + k * 2048, 8192, 1024)
                                     : sdesc_sw128(sA + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(sB + k * 2048, 8192, 1024)
                                     : sdesc_sw128(sB + k * 32, 16, 1024);
            tc_mma_bf16(d, ad, bd, IDESC, (kb > w.kb_begin || k > 0) ? 1u : 0u);
          }
          any = true;
          tc_commit(bar_s(EMPTY + stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(bar_s(TFULL + acc));
        acc ^= 1;
        if (acc == 0) aphase ^= 1u;
      }
      if (!ok) {
        record_timeout(p, abort_flag);
        if (any) {  // wait for the MMAs already issued before TMEM is freed
          tc_commit(bar_s(DRAIN));
          volatile int never = 0;
          mbar_wait(bar_s(DRAIN), 0, 10000000ull, &never);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int row_in_tile = q * 32 + lane;
    int slot = 0;
    uint32_t sphase = 0;
    int acc = 0;
    uint32_t aphase = 0;
    while (true) {
      if (!mbar_wait(bar_s(SFULL + slot), sphase, lim, abort_flag)) {
        record_timeout(p, abort_flag);
        break;
      }
      const int unit = sched[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_s(SEMPTY + slot));
      if (++slot == SCHED_SLOTS) { slot = 0; sphase ^= 1u; }
      if (unit < 0) break;
      const Work w = decode_unit(p, unit);
      const Prob& P = p.prob[w.prob];
      if (!mbar_wait(bar_s(TFULL + acc), aphase, lim, abort_flag)) {
        record_timeout(p, abort_flag);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + acc * MMA_N + (static_cast<uint32_t>(q * 32) << 16);
      const int row = w.tm * BM + row_in_tile;
      const int col0 = w.tn * TILE_N;
      if constexpr (EPI == EPI_GATED_FWD) {
        epi_gated_fwd<ACT_SILU>(p, P, tb, row, col0);
      } else if constexpr (EPI == EPI_ACT_FWD) {
        if (p.act == ACT_RELU_SQ) epi_act_fwd<ACT_RELU_SQ>(p, P, tb, row, col0);
        else epi_act_fwd<ACT_GELU_TANH>(p, P, tb, row, col0);
      } else if constexpr (EPI == EPI_DGATED) {
        epi_dact<ACT_SILU, true>(p, P, tb, row, col0);
      } else if constexpr (EPI == EPI_DACT) {
        if (p.act == ACT_RELU_SQ) epi_dact<ACT_RELU_SQ, false>(p, P, tb, row, col0);
        else epi_dact<ACT_GELU_TANH, false>(p, P, tb, row, col0);
      } else {
        epi_plain<EPI>(P, tb, row, col0);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_s(TEMPTY + acc));
      acc ^= 1;
      if (acc == 0) aphase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int EPI, bool A_MN, bool B_MN>
cudaError_t launch_gemm(const Params& p, int grid, cudaStream_t stream, bool pdl) {
  auto kern = k_mlp_gemm<EPI, A_MN, B_MN>;
  static std::atomic<unsigned> configured_dev_mask{0};  // devices that got the smem attribute
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 31 || !(configured_dev_mask.load() & (1u << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 31) configured_dev_mask.fetch_or(1u << dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace mlpk
