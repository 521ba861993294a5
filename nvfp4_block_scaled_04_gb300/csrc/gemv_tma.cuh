// TMA-fed variant of the skinny W4A16 kernel (decode GEMV and the MoE expert
// GEMMs): the same arithmetic as gemv_core.cuh, with memory decoupled from
// compute.
//
// One CTA = 8 consumer warps (16 weight rows each, 128 rows) + 1 producer
// warp. The producer streams, per stage of 256 K-elements,
//   - the 128 rows x 128 bytes of packed codes with one 2-D TMA copy (128B
//     swizzle, so the consumers' 16-byte fragment reads spread over the
//     banks),
//   - the rows' 16 block scales per row with a second 2-D TMA copy,
//   - the activation fragments of the stage with 1-D bulk copies,
// into a 3- or 4-stage shared-memory ring (mbarrier full/empty pairs). The
// weights of the first stages are requested before the kernel waits on the
// activation prep (programmatic dependent launch), so the prep's latency
// hides behind the weight stream. With split-K, every CTA writes fp32
// partials to the workspace and the last CTA of a tile to arrive (an atomic
// counter) sums them in split order, so the result is deterministic and no
// thread-block cluster has to fit on one GPC.
#pragma once

#include "gemv_core.cuh"
#include "tc_util.cuh"

namespace nvfp4 {

// MT m-tiles (16 rows each) per consumer warp: 8 / MT row groups cover the
// CTA's 128 rows, and every activation fragment read from shared memory feeds
// MT MMAs. KW warps share a row group, each taking one of the stage's two
// K-iterations (KW = 2) or both (KW = 1): more warps per SM to hide latency
// at the same shared memory.
template <int MT, int KW>
struct GtWarps {
  static constexpr int GROUPS = 8 / MT;
  static constexpr int CONSUMERS = GROUPS * KW;
  static constexpr int THREADS = (CONSUMERS + 1) * 32;
};
constexpr int GT_CODES = 128 * 128;      // one stage of codes: 128 rows x 128 bytes
constexpr int GT_SCALES = 128 * 16;      // one stage of scales: 128 rows x 16 bytes

template <int NT>
struct GtCfg {
  static constexpr int XB = 2 * NT * 2048;                                    // activations of 2 iterations
  static constexpr int STAGE = (GT_CODES + GT_SCALES + XB + 1023) / 1024 * 1024;
  static constexpr int STAGES = NT <= 2 ? 4 : 3;
  static constexpr int RING = STAGES * STAGE;
  static constexpr int SMEM = RING + 1024 /*alignment*/ + 512 /*barriers, shifts, flags*/;
};

struct TmaSkinnyParams {
  const float* s_t;
  int64_t K;
  int64_t n_rows;              // PLAIN: N
  const uint4* xfrag;
  const int* pexp;
  int64_t M;
  int split;
  uint16_t* Y;
  const int* chunk_count;
  const int* chunk_expert;
  const int* chunk_rows;
  int64_t inter;
  int64_t hidden;
  int64_t rows_per_expert;
  uint16_t* h_out;
  float* y_out;
  int* status;
  float* partials;             // split-K > 1: [tile][split][32 tokens][128 rows] fp32
  unsigned int* counters;      // split-K > 1: one arrival counter per tile, zeroed by the prep kernel
};

// MMA row g of a warp's 16-row tile reads shared-memory row sigma(g) (and
// sigma(g) + 8): lanes of one 8-lane phase (g = 2q, 2q+1) then read rows that
// differ in bit 2, whose 128B-swizzled chunks never share banks.
NVFP4_DEV int gt_sigma(int g) { return ((g & 1) << 2) | (g >> 1); }

NVFP4_DEV uint32_t lds_u16(uint32_t saddr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr));
  return v;
}
NVFP4_DEV uint4 lds_v4(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(saddr));
  return v;
}

// One K-iteration (128 K) of a stage: the warp's MT m-tiles of 16 weight rows
// (row group grp) against NT n-tiles of 8 tokens; j selects the iteration
// within the stage (codes at 16-byte chunks 4j..4j+3 of each 128-byte row,
// scales at bytes 8j..8j+7, activation fragments at j * NT * 2048).
template <int NT, int MT>
NVFP4_DEV void gt_mma_iteration(uint32_t stage, int j, int grp, int sw, int t, int lane, float (&acc)[MT][NT][4]) {
  const uint32_t phys = static_cast<uint32_t>(((4 * j + t) ^ sw) << 4);
  uint32_t wa[MT][4], wb[MT][4], sa[MT][2], sb[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int rl = (grp * MT + mt) * 16 + sw;
    const uint4 ca = lds_v4(stage + rl * 128 + phys);
    const uint4 cb = lds_v4(stage + (rl + 8) * 128 + phys);
    wa[mt][0] = ca.x; wa[mt][1] = ca.y; wa[mt][2] = ca.z; wa[mt][3] = ca.w;
    wb[mt][0] = cb.x; wb[mt][1] = cb.y; wb[mt][2] = cb.z; wb[mt][3] = cb.w;
    const uint32_t scA = e4m3x2_to_f16x2(lds_u16(stage + GT_CODES + rl * 16 + 8 * j + 2 * t));
    const uint32_t scB = e4m3x2_to_f16x2(lds_u16(stage + GT_CODES + (rl + 8) * 16 + 8 * j + 2 * t));
    sa[mt][0] = dup_lo(scA); sa[mt][1] = dup_hi(scA);
    sb[mt][0] = dup_lo(scB); sb[mt][1] = dup_hi(scB);
  }
  const uint32_t xs = stage + GT_CODES + GT_SCALES + j * NT * 2048 + lane * 16;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t A0[MT][4], A1[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t fa[4], fb[4];
      e2m1x8_to_f16x2(wa[mt][w], fa);
      e2m1x8_to_f16x2(wb[mt][w], fb);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        fa[e] = hmul2(fa[e], sa[mt][w >> 1]);
        fb[e] = hmul2(fb[e], sb[mt][w >> 1]);
      }
      A0[mt][0] = fa[0]; A0[mt][1] = fb[0]; A0[mt][2] = fa[1]; A0[mt][3] = fb[1];
      A1[mt][0] = fa[2]; A1[mt][1] = fb[2]; A1[mt][2] = fa[3]; A1[mt][3] = fb[3];
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint4 bx = lds_v4(xs + (nt * 4 + w) * 512);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        mma_f16_16816(acc[mt][nt], A0[mt], bx.x, bx.y);
        mma_f16_16816(acc[mt][nt], A1[mt], bx.z, bx.w);
      }
    }
  }
}

template <int NT, int MODE, int MT, int KW>
__global__ void __launch_bounds__(GtWarps<MT, KW>::THREADS, 2)
    skinny_tma_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_scales,
                      const TmaSkinnyParams p) {
  using C = GtCfg<NT>;
  pdl_launch_dependents();   // the next call's activation prep may queue up now
  constexpr int NCW = GtWarps<MT, KW>::CONSUMERS;
  constexpr int NGR = GtWarps<MT, KW>::GROUPS;
  constexpr int NTHR = GtWarps<MT, KW>::THREADS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  uint8_t* ring_ptr = smem_raw + (ring - raw);
  const uint32_t bar_base = ring + C::RING;
  int* pexp_s = reinterpret_cast<int*>(ring_ptr + C::RING + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ring_ptr + C::RING + 64 + 128);
  int* s_last = reinterpret_cast<int*>(ring_ptr + C::RING + 64 + 132);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::STAGES + s); };

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int S = p.split;
  const int s = (MODE == SK_PLAIN) ? static_cast<int>(blockIdx.x) : 0;
  const int64_t n_it = p.K / GV_KIT;
  const int64_t n_st_total = (n_it + 1) / 2;
  const int st0 = static_cast<int>(n_st_total * s / S);
  const int n_st = static_cast<int>(n_st_total * (s + 1) / S) - st0;
  const int64_t it0 = 2LL * st0;
  const int64_t it_end_raw = 2LL * (st0 + n_st);
  const int64_t it_end = it_end_raw < n_it ? it_end_raw : n_it;

  int64_t chunk, row_tile;
  int rows_in_chunk;
  int expert = 0;
  if (MODE == SK_MOE_GATEUP || MODE == SK_MOE_DOWN) {
    chunk = blockIdx.x;
    row_tile = blockIdx.y;
    if (chunk >= *p.chunk_count) return;
    expert = p.chunk_expert[chunk];
    rows_in_chunk = p.chunk_rows[chunk];
  } else {
    chunk = blockIdx.z;
    row_tile = blockIdx.y;
    const int64_t left = p.M - chunk * GV_MCHUNK;
    rows_in_chunk = static_cast<int>(left < GV_MCHUNK ? left : GV_MCHUNK);
  }

  if (tid == 0) {
    for (int q = 0; q < C::STAGES; ++q) {
      mbar_init(full_bar(q), 1);
      mbar_init(empty_bar(q), NCW);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_codes) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_scales) : "memory");
  }
  __syncthreads();

  float acc[MT][NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;

  int issued = 0;
  if (warp == NCW) {
    if (lane == 0) {
      // y coordinates of the tile's rows in the stacked weight
      int y_a, y_b = 0;
      if (MODE == SK_MOE_GATEUP) {
        y_a = static_cast<int>(expert * p.rows_per_expert + row_tile * 64);
        y_b = static_cast<int>(expert * p.rows_per_expert + p.inter + row_tile * 64);
      } else if (MODE == SK_MOE_DOWN) {
        y_a = static_cast<int>(expert * p.rows_per_expert + row_tile * GV_ROWS);
      } else {
        y_a = static_cast<int>(row_tile * GV_ROWS);
      }
      auto x_iters = [&](int st) {
        const int64_t a = it0 + 2LL * st;
        const int64_t left = it_end - a;
        return static_cast<int>(left < 2 ? left : 2);
      };
      auto issue_weights = [&](int st) {
        const int q = st % C::STAGES;
        const uint32_t stage = ring + q * C::STAGE;
        const uint32_t bytes = GT_CODES + GT_SCALES + x_iters(st) * NT * 2048 + (st == 0 ? 128u : 0u);
        mbar_arrive_expect_tx(full_bar(q), bytes);
        const int xc = static_cast<int>((it0 + 2LL * st) * 64);
        const int xs = static_cast<int>((it0 + 2LL * st) * 8);
        if (MODE == SK_MOE_GATEUP) {
          tma_load_2d(stage, &map_codes, xc, y_a, full_bar(q));
          tma_load_2d(stage + GT_CODES / 2, &map_codes, xc, y_b, full_bar(q));
          tma_load_2d(stage + GT_CODES, &map_scales, xs, y_a, full_bar(q));
          tma_load_2d(stage + GT_CODES + GT_SCALES / 2, &map_scales, xs, y_b, full_bar(q));
        } else {
          tma_load_2d(stage, &map_codes, xc, y_a, full_bar(q));
          tma_load_2d(stage + GT_CODES, &map_scales, xs, y_a, full_bar(q));
        }
      };
      auto issue_x = [&](int st) {
        const int q = st % C::STAGES;
        const uint32_t stage = ring + q * C::STAGE;
        if (st == 0) bulk_load(smem_addr(pexp_s), p.pexp + chunk * GV_MCHUNK, 128u, full_bar(q));
        for (int j = 0; j < x_iters(st); ++j) {
          const uint4* src = p.xfrag + xfrag_unit(chunk, n_it, it0 + 2LL * st + j, 0, 0, 0);
          bulk_load(stage + GT_CODES + GT_SCALES + j * NT * 2048, src, NT * 2048u, full_bar(q));
        }
      };
      const int pre = n_st < C::STAGES ? n_st : C::STAGES;
      for (int st = 0; st < pre; ++st) issue_weights(st);
      pdl_wait();   // the activation prep has finished and its writes are visible
      for (int st = 0; st < pre; ++st) issue_x(st);
      issued = pre;
      for (int st = pre; st < n_st; ++st) {
        const int q = st % C::STAGES;
        if (!mbar_wait_bounded(empty_bar(q), ((st / C::STAGES) - 1) & 1, abort_flag, p.status)) break;
        issue_weights(st);
        issue_x(st);
        ++issued;
      }
    }
  } else {
    const int sw = gt_sigma(g);               // smem row (mod 8) of MMA row g
    const int grp = warp % NGR;               // row group of this warp
    const int jk = warp / NGR;                // its K-iteration within a stage when KW == 2
    for (int st = 0; st < n_st; ++st) {
      const int q = st % C::STAGES;
      if (!mbar_wait_bounded(full_bar(q), (st / C::STAGES) & 1, abort_flag, p.status)) break;
      const uint32_t stage = ring + q * C::STAGE;
#pragma unroll
      for (int jj = 0; jj < 3 - KW; ++jj) {
        const int j = KW == 2 ? jk : jj;
        if (it0 + 2LL * st + j < it_end) {
          gt_mma_iteration<NT, MT>(stage, j, grp, sw, t, lane, acc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(q));
    }
  }
  // after a give-up, let copies already in flight land before the ring is reused
  if (warp == NCW && lane == 0 && *abort_flag) {
    const int first = issued > C::STAGES ? issued - C::STAGES : 0;
    for (int st = first; st < issued; ++st)
      mbar_wait_bounded(full_bar(st % C::STAGES), (st / C::STAGES) & 1, nullptr, p.status, 100000000ull);
  }
  __syncthreads();   // the ring is free: it now holds this CTA's partial sums
  // KW slices of [8*NT tokens][128 rows] fp32, one per K-iteration half
  float* part = reinterpret_cast<float*>(ring_ptr);
  if (warp < NCW) {
    const int grp = warp % NGR, jk = warp / NGR;
    float* slice = part + jk * (8 * NT * GV_ROWS);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          slice[(nt * 8 + 2 * t + (e & 1)) * GV_ROWS + (grp * MT + mt) * 16 + gt_sigma(g) + 8 * (e >> 1)] =
              acc[mt][nt][e];
  }
  __syncthreads();
  auto psum = [&](int tok, int r) {
    float v = part[tok * GV_ROWS + r];
    if (KW == 2) v += part[8 * NT * GV_ROWS + tok * GV_ROWS + r];
    return v;
  };
  const int64_t row_base = chunk * GV_MCHUNK;
  const float st = p.s_t[expert];
  if (S == 1) {
    const int width = (MODE == SK_MOE_GATEUP) ? 64 : GV_ROWS;
    for (int e = tid; e < rows_in_chunk * width; e += NTHR) {
      const int tok = e / width;
      const int r = e % width;
      const float v = psum(tok, r);
      const float mul = ldexpf(st, pexp_s[tok]);
      if (MODE == SK_PLAIN) {
        const int64_t n = row_tile * GV_ROWS + r;
        if (n < p.n_rows) p.Y[(row_base + tok) * p.n_rows + n] = static_cast<uint16_t>(f32_to_bf16_bits(v * mul));
      } else if (MODE == SK_MOE_GATEUP) {
        const float gg = v * mul;
        const float uu = psum(tok, 64 + r) * mul;
        const float hh = gg / (1.0f + expf(-gg)) * uu;
        p.h_out[(row_base + tok) * p.inter + row_tile * 64 + r] = static_cast<uint16_t>(f32_to_bf16_bits(hh));
      } else {
        const int64_t c = row_tile * GV_ROWS + r;
        if (c < p.hidden) p.y_out[(row_base + tok) * p.hidden + c] = v * mul;
      }
    }
  } else if (MODE == SK_PLAIN) {
    // split-K: partials to global memory, the last CTA of the tile reduces
    const int64_t tile = chunk * gridDim.y + row_tile;
    float* mine = p.partials + ((tile * S + s) * GV_MCHUNK) * GV_ROWS;
    for (int e = tid; e < rows_in_chunk * GV_ROWS; e += NTHR) mine[e] = psum(e / GV_ROWS, e % GV_ROWS);
    __threadfence();
    __syncthreads();
    if (tid == 0) *s_last = atomicAdd(&p.counters[tile], 1u) == static_cast<unsigned>(S - 1);
    __syncthreads();
    if (*s_last) {
      __threadfence();
      const float* all = p.partials + (tile * S * GV_MCHUNK) * GV_ROWS;
      for (int e = tid; e < rows_in_chunk * GV_ROWS; e += NTHR) {
        const int tok = e / GV_ROWS;
        const int r = e % GV_ROWS;
        // all S (<= 8) partials in flight at once, summed in split order
        float x[8];
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) x[qq] = qq < S ? __ldcg(all + (qq * GV_MCHUNK + tok) * GV_ROWS + r) : 0.f;
        float v = 0.f;
#pragma unroll
        for (int qq = 0; qq < 8; ++qq)
          if (qq < S) v += x[qq];
        const int64_t n = row_tile * GV_ROWS + r;
        if (n < p.n_rows)
          p.Y[(row_base + tok) * p.n_rows + n] =
              static_cast<uint16_t>(f32_to_bf16_bits(v * ldexpf(st, pexp_s[tok])));
      }
    }
  }
}

}  // namespace nvfp4
