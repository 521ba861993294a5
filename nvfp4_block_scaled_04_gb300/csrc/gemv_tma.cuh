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

// Scales of gathered rows: tile::gather4 writes a lane's four 16-byte rows
// to one 128-byte-aligned slot (a tensor copy's shared-memory destination
// must be 128-byte aligned), so row r sits at (r / 4) * 128 + (r % 4) * 16.
constexpr int GT_SCALES_GATHERED = 128 * 32;

template <bool GATHERED>
NVFP4_DEV uint32_t gt_scale_row(int r) {
  return GATHERED ? static_cast<uint32_t>((r >> 2) * 128 + (r & 3) * 16) : static_cast<uint32_t>(r * 16);
}

template <int NT, int SC = GT_SCALES>
struct GtCfg {
  static constexpr int SCALES = SC;                                           // scale area of a stage
  static constexpr int XB = 2 * NT * 2048;                                    // activations of 2 iterations
  static constexpr int STAGE = (GT_CODES + SC + XB + 1023) / 1024 * 1024;
  static constexpr int STAGES = NT <= 2 ? 4 : 3;
  static constexpr int RING = STAGES * STAGE;
  static constexpr int SMEM = RING + 1024 /*alignment*/ + 1024 /*barriers, shifts, flags, argmax ids*/;
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
  uint16_t* y_out;             // MOE_DOWN: bf16 [padded rows][H]
  int* status;
  float* partials;             // split-K > 1: [tile][split][32 tokens][128 rows] fp32
  unsigned int* counters;      // split-K > 1: one arrival counter per tile, zeroed by the prep kernel
  int weights_once;            // MoE: each weight byte is read once per call (evict-first L2 policy)
  // ARGMAX (split 1): candidate j is weight row idx[j] (row j when idx is null)
  const int32_t* idx;
  int64_t w_rows;              // rows gathered in place: rows of the weight; an idx entry outside
                               // [0, w_rows) is skipped (compact rows: 0, idx holds labels only)
  unsigned long long* keys;    // [M] best (logit order key, ~id) so far, zero on entry
  unsigned int* counter;       // finished CTAs, zero on entry
  int32_t* out_ids;
  float* out_logit;            // nullable
  const uint8_t* codes;        // row-streaming ARGMAX: the weight itself
  const uint8_t* scales;
  // ARGMAX as a speculative verify head (n_accepted non-null): the M rows are
  // `M / (n_draft + 1)` sequences of n_draft + 1 positions; the finishing CTA
  // also counts, per sequence, the leading drafts equal to the argmax at
  // their position
  const int32_t* draft_ids;    // [M / (n_draft + 1)][n_draft]
  int n_draft;
  int32_t* n_accepted;         // [M / (n_draft + 1)]
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
// scales at bytes 8j..8j+7, activation fragments at j * NT * 2048). Only the
// first nt_active n-tiles hold tokens (a partly filled chunk, e.g. an expert
// with few routed rows); the MMAs of the others are skipped.
template <int NT, int MT, bool GATHERED = false>
NVFP4_DEV void gt_mma_iteration(uint32_t stage, int j, int grp, int sw, int t, int lane, int nt_active,
                                float (&acc)[MT][NT][4]) {
  constexpr int SC = GATHERED ? GT_SCALES_GATHERED : GT_SCALES;
  const uint32_t phys = static_cast<uint32_t>(((4 * j + t) ^ sw) << 4);
  uint32_t wa[MT][4], wb[MT][4], sa[MT][2], sb[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int rl = (grp * MT + mt) * 16 + sw;
    const uint4 ca = lds_v4(stage + rl * 128 + phys);
    const uint4 cb = lds_v4(stage + (rl + 8) * 128 + phys);
    wa[mt][0] = ca.x; wa[mt][1] = ca.y; wa[mt][2] = ca.z; wa[mt][3] = ca.w;
    wb[mt][0] = cb.x; wb[mt][1] = cb.y; wb[mt][2] = cb.z; wb[mt][3] = cb.w;
    const uint32_t scA = e4m3x2_to_f16x2(lds_u16(stage + GT_CODES + gt_scale_row<GATHERED>(rl) + 8 * j + 2 * t));
    const uint32_t scB = e4m3x2_to_f16x2(lds_u16(stage + GT_CODES + gt_scale_row<GATHERED>(rl + 8) + 8 * j + 2 * t));
    sa[mt][0] = dup_lo(scA); sa[mt][1] = dup_hi(scA);
    sb[mt][0] = dup_lo(scB); sb[mt][1] = dup_hi(scB);
  }
  const uint32_t xs = stage + GT_CODES + SC + j * NT * 2048 + lane * 16;
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
      if (nt < nt_active) {
        const uint4 bx = lds_v4(xs + (nt * 4 + w) * 512);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_f16_16816(acc[mt][nt], A0[mt], bx.x, bx.y);
          mma_f16_16816(acc[mt][nt], A1[mt], bx.z, bx.w);
        }
      }
    }
  }
}

// GATHER (ARGMAX with an index only): weight rows come in by tile::gather4;
// otherwise by 2-D boxes of consecutive rows.
template <int NT, int MODE, int MT, int KW, bool GATHER = false>
__global__ void __launch_bounds__(GtWarps<MT, KW>::THREADS, 2)
    skinny_tma_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_scales,
                      const TmaSkinnyParams p) {
  constexpr bool GATHERED = MODE == SK_ARGMAX && GATHER;
  // a tile of 64 gate rows and the matching 64 up rows, SiLU * mul fused
  constexpr bool GATEUP = MODE == SK_MOE_GATEUP || MODE == SK_GATEUP_DENSE;
  using C = GtCfg<NT, GATHERED ? GT_SCALES_GATHERED : GT_SCALES>;
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
  unsigned long long* kbest = reinterpret_cast<unsigned long long*>(ring_ptr + C::RING + 256);   // ARGMAX, [32]
  int* sidx = reinterpret_cast<int*>(ring_ptr + C::RING + 512);   // ARGMAX: vocabulary ids of the tile's rows, [128]
  static_assert(2 * C::STAGES * 8 <= 64, "barrier area");
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::STAGES + s); };

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int S = p.split;
  const int s = (MODE == SK_PLAIN || MODE == SK_GATEUP_DENSE) ? static_cast<int>(blockIdx.x) : 0;
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
  if (MODE == SK_ARGMAX && tid < GV_MCHUNK) kbest[tid] = 0ull;
  __syncthreads();

  float acc[MT][NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;

  int issued = 0;
  if (GATHERED && warp == NCW) {
    // Gathered rows: lane l loads candidate rows 4l .. 4l+3 of the tile with
    // one tile::gather4 per stage for the codes (4 x 128 bytes, 128B swizzle,
    // so they land exactly where a 2-D box would put them) and one for the
    // scales (4 x 16 bytes). Candidates past the end repeat the last row;
    // the epilogue ignores them.
    int rid[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t j0 = row_tile * GV_ROWS + 4 * lane + i;
      const int64_t j = j0 < p.n_rows ? j0 : p.n_rows - 1;
      rid[i] = p.idx ? p.idx[j] : static_cast<int>(j);
      if (rid[i] < 0 || rid[i] >= p.w_rows) rid[i] = 0;   // a skipped entry reads row 0; its key is dropped
    }
    auto issue_weights = [&](int st) {
      const int q = st % C::STAGES;
      const uint32_t stage = ring + q * C::STAGE;
      // bytes that land: 32 lanes x (4 x 128 code bytes + 4 x 16 scale bytes)
      if (lane == 0)
        mbar_arrive_expect_tx(full_bar(q), GT_CODES + GT_SCALES + 2 * NT * 2048 + (st == 0 ? 128u : 0u));
      __syncwarp();
      const int xc = static_cast<int>((it0 + 2LL * st) * 64);
      const int xs = static_cast<int>((it0 + 2LL * st) * 8);
      tma_gather4(stage + lane * 512, &map_codes, xc, rid[0], rid[1], rid[2], rid[3], full_bar(q));
      tma_gather4(stage + GT_CODES + lane * 128, &map_scales, xs, rid[0], rid[1], rid[2], rid[3], full_bar(q));
    };
    auto issue_x = [&](int st) {
      const int q = st % C::STAGES;
      const uint32_t stage = ring + q * C::STAGE;
      if (st == 0) bulk_load(smem_addr(pexp_s), p.pexp + chunk * GV_MCHUNK, 128u, full_bar(q));
#pragma unroll
      for (int j = 0; j < 2; ++j)
        bulk_load(stage + GT_CODES + C::SCALES + j * NT * 2048,
                  p.xfrag + xfrag_unit(chunk, n_it, it0 + 2LL * st + j, 0, 0, 0), NT * 2048u, full_bar(q));
    };
    // Stages go out in pairs: a lane requests K-chunks st and st + 1 of its
    // four rows back to back, 256 contiguous bytes per row, so the random
    // rows cost one DRAM page opening per 256 bytes instead of per 128.
    const int pre = n_st < C::STAGES ? n_st : C::STAGES;
    for (int st = 0; st < pre; ++st) issue_weights(st);
    pdl_wait();   // the activation prep has finished and its writes are visible
    if (lane == 0)
      for (int st = 0; st < pre; ++st) issue_x(st);
    issued = pre;
    for (int st = pre; st < n_st; st += 2) {
      const int n = st + 1 < n_st ? 2 : 1;
      bool ok = true;
      for (int u = 0; u < n && ok; ++u) {
        const int q = (st + u) % C::STAGES;
        ok = __all_sync(0xffffffffu,
                        mbar_wait_bounded(empty_bar(q), (((st + u) / C::STAGES) - 1) & 1, abort_flag, p.status));
      }
      if (!ok) break;
      for (int u = 0; u < n; ++u) issue_weights(st + u);
      if (lane == 0)
        for (int u = 0; u < n; ++u) issue_x(st + u);
      issued += n;
    }
  } else if (warp == NCW) {
    if (lane == 0) {
      // y coordinates of the tile's rows in the stacked weight
      int y_a, y_b = 0;
      if (MODE == SK_MOE_GATEUP) {
        y_a = static_cast<int>(expert * p.rows_per_expert + row_tile * 64);
        y_b = static_cast<int>(expert * p.rows_per_expert + p.inter + row_tile * 64);
      } else if (MODE == SK_GATEUP_DENSE) {
        y_a = static_cast<int>(row_tile * 64);
        y_b = static_cast<int>(p.inter + row_tile * 64);
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
        // a weight byte read once per call is evicted from L2 first (measured:
        // decode step 183 -> 177 us, MoE layer at 256 tokens 173 -> 167 us);
        // routed experts with several token chunks re-read theirs
        const bool once = MODE == SK_PLAIN || MODE == SK_ARGMAX || MODE == SK_GATEUP_DENSE || p.weights_once;
        if (GATEUP && once) {
          const uint64_t pol = l2_policy_evict_first();
          tma_load_2d_hint(stage, &map_codes, xc, y_a, full_bar(q), pol);
          tma_load_2d_hint(stage + GT_CODES / 2, &map_codes, xc, y_b, full_bar(q), pol);
          tma_load_2d_hint(stage + GT_CODES, &map_scales, xs, y_a, full_bar(q), pol);
          tma_load_2d_hint(stage + GT_CODES + GT_SCALES / 2, &map_scales, xs, y_b, full_bar(q), pol);
        } else if (GATEUP) {
          tma_load_2d(stage, &map_codes, xc, y_a, full_bar(q));
          tma_load_2d(stage + GT_CODES / 2, &map_codes, xc, y_b, full_bar(q));
          tma_load_2d(stage + GT_CODES, &map_scales, xs, y_a, full_bar(q));
          tma_load_2d(stage + GT_CODES + GT_SCALES / 2, &map_scales, xs, y_b, full_bar(q));
        } else if (once) {
          const uint64_t pol = l2_policy_evict_first();
          tma_load_2d_hint(stage, &map_codes, xc, y_a, full_bar(q), pol);
          tma_load_2d_hint(stage + GT_CODES, &map_scales, xs, y_a, full_bar(q), pol);
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
    if (MODE == SK_ARGMAX && tid < GV_ROWS) {
      // the epilogue's row ids, fetched while the first stages are in flight
      const int64_t j = row_tile * GV_ROWS + tid;
      sidx[tid] = j < p.n_rows ? (p.idx ? p.idx[j] : static_cast<int>(j)) : 0;
    }
    const int sw = gt_sigma(g);               // smem row (mod 8) of MMA row g
    const int grp = warp % NGR;               // row group of this warp
    const int jk = warp / NGR;                // its K-iteration within a stage when KW == 2
    const int nt_active = (rows_in_chunk + 7) / 8;
    for (int st = 0; st < n_st; ++st) {
      const int q = st % C::STAGES;
      if (!mbar_wait_bounded(full_bar(q), (st / C::STAGES) & 1, abort_flag, p.status)) break;
      const uint32_t stage = ring + q * C::STAGE;
#pragma unroll
      for (int jj = 0; jj < 3 - KW; ++jj) {
        const int j = KW == 2 ? jk : jj;
        if (it0 + 2LL * st + j < it_end) {
          gt_mma_iteration<NT, MT, GATHERED>(stage, j, grp, sw, t, lane, nt_active, acc);
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
    const int width = GATEUP ? 64 : GV_ROWS;
    // ARGMAX: the loop runs warp-uniformly over whole rounds of NTHR, so each
    // round's keys can meet in a warp maximum before one shared atomic per
    // warp and token (a 128-byte row of outputs belongs to one token)
    const int n_out = rows_in_chunk * width;
    const int n_loop = MODE == SK_ARGMAX ? (n_out + NTHR - 1) / NTHR * NTHR : n_out;
    for (int e = tid; e < n_loop; e += NTHR) {
      unsigned long long key = 0ull;
      int key_tok = -1;
      if (e < n_out) {
        const int tok = e / width;
        const int r = e % width;
        const float v = psum(tok, r);
        const float mul = ldexpf(st, pexp_s[tok]);
        if (MODE == SK_PLAIN) {
          const int64_t n = row_tile * GV_ROWS + r;
          if (n < p.n_rows) p.Y[(row_base + tok) * p.n_rows + n] = static_cast<uint16_t>(f32_to_bf16_bits(v * mul));
        } else if (MODE == SK_ARGMAX) {
          // key: logit order first, then the lower vocabulary id
          const int64_t j = row_tile * GV_ROWS + r;
          if (j < p.n_rows && (!GATHERED || (sidx[r] >= 0 && sidx[r] < p.w_rows))) {
            const uint32_t vid = static_cast<uint32_t>(sidx[r]);
            key = (static_cast<unsigned long long>(float_order_key(v * mul)) << 32) | (0xFFFFFFFFu - vid);
          }
          key_tok = tok;   // set for rows past the end too: the groups below follow the output index
        } else if (GATEUP) {
          const float gg = v * mul;
          const float uu = psum(tok, 64 + r) * mul;
          const float hh = gg / (1.0f + expf(-gg)) * uu;
          p.h_out[(row_base + tok) * p.inter + row_tile * 64 + r] = static_cast<uint16_t>(f32_to_bf16_bits(hh));
        } else {
          const int64_t c = row_tile * GV_ROWS + r;
          if (c < p.hidden) p.y_out[(row_base + tok) * p.hidden + c] = static_cast<uint16_t>(f32_to_bf16_bits(v * mul));
        }
      }
      if (MODE == SK_ARGMAX) {
        // lanes of a warp cover consecutive outputs: one or two tokens per warp
        // and round (a row of outputs is 128 wide), then lanes past the end
        const int tok_lo = __shfl_sync(0xffffffffu, key_tok, 0);
#pragma unroll
        for (int side = 0; side < 2; ++side) {
          unsigned long long k = (side == 0) == (key_tok == tok_lo) ? key : 0ull;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, k, o);
            k = other > k ? other : k;
          }
          const int kt = side == 0 ? tok_lo : __shfl_sync(0xffffffffu, key_tok, 31);
          if (lane == 0 && kt >= 0 && k != 0ull && (side == 0 || kt != tok_lo)) atomicMax(&kbest[kt], k);
        }
      }
    }
    if (MODE == SK_ARGMAX) {
      // this CTA's per-token best into the global keys; the last CTA to
      // finish reads them out and leaves keys and counter at zero
      __syncthreads();
      if (tid < rows_in_chunk) atomicMax(&p.keys[row_base + tid], kbest[tid]);
      fence_acq_rel_gpu();
      __syncthreads();
      if (tid == 0) *s_last = atomicAdd(p.counter, 1u) == gridDim.x * gridDim.y * gridDim.z - 1;
      __syncthreads();
      if (*s_last) {
        fence_acq_rel_gpu();
        for (int64_t m = tid; m < p.M; m += NTHR) {
          const unsigned long long key = atomicExch(&p.keys[m], 0ull);
          p.out_ids[m] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
          if (p.out_logit) p.out_logit[m] = float_from_order_key(static_cast<uint32_t>(key >> 32));
        }
        if (tid == 0) atomicExch(p.counter, 0u);
        if (p.n_accepted) {
          // greedy acceptance: the drafts of a sequence are accepted up to the
          // first one that differs from the argmax at its position
          __syncthreads();   // this CTA's writes of out_ids are visible to it
          const int d1 = p.n_draft + 1;
          for (int b = tid; b < static_cast<int>(p.M) / d1; b += NTHR) {
            int n = 0;
            while (n < p.n_draft && p.draft_ids[b * p.n_draft + n] == p.out_ids[b * d1 + n]) ++n;
            p.n_accepted[b] = n;
          }
        }
      }
    }
  } else if (MODE == SK_PLAIN || MODE == SK_GATEUP_DENSE) {
    // split-K: partials to global memory, the last CTA of the tile reduces
    const int64_t tile = chunk * gridDim.y + row_tile;
    constexpr int P4 = GV_MCHUNK * GV_ROWS / 4;   // float4 groups of one split's partial
    float4* mine = reinterpret_cast<float4*>(p.partials) + (tile * S + s) * P4;
    const int n4 = rows_in_chunk * (GV_ROWS / 4);  // groups in use: [token][128 rows / 4]
    for (int e4 = tid; e4 < n4; e4 += NTHR) {
      const int tok = e4 >> 5, r = (e4 & 31) * 4;
      mine[e4] = make_float4(psum(tok, r), psum(tok, r + 1), psum(tok, r + 2), psum(tok, r + 3));
    }
    fence_acq_rel_gpu();
    __syncthreads();
    if (tid == 0) *s_last = atomicAdd(&p.counters[tile], 1u) == static_cast<unsigned>(S - 1);
    __syncthreads();
    if (MODE == SK_GATEUP_DENSE && *s_last) {
      // gate rows r .. r + 3 are float4 group tok * 32 + r / 4, the matching
      // up rows group tok * 32 + 16 + r / 4; both summed in split order
      fence_acq_rel_gpu();
      const float4* all = reinterpret_cast<const float4*>(p.partials) + tile * S * P4;
      const int n4g = rows_in_chunk * 16;
      for (int e = tid; e < n4g; e += NTHR) {
        const int tok = e >> 4, gi = tok * 32 + (e & 15);
        float4 xg[8], xu[8];
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          xg[qq] = qq < S ? __ldcg(all + qq * P4 + gi) : make_float4(0.f, 0.f, 0.f, 0.f);
          xu[qq] = qq < S ? __ldcg(all + qq * P4 + gi + 16) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float g4[4] = {0.f, 0.f, 0.f, 0.f}, u4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int qq = 0; qq < 8; ++qq)
          if (qq < S) {
            g4[0] += xg[qq].x; g4[1] += xg[qq].y; g4[2] += xg[qq].z; g4[3] += xg[qq].w;
            u4[0] += xu[qq].x; u4[1] += xu[qq].y; u4[2] += xu[qq].z; u4[3] += xu[qq].w;
          }
        const float mul = ldexpf(st, pexp_s[tok]);
        float h4[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float gg = g4[c] * mul, uu = u4[c] * mul;
          h4[c] = gg / (1.0f + expf(-gg)) * uu;
        }
        *reinterpret_cast<uint2*>(p.h_out + (row_base + tok) * p.inter + row_tile * 64 + (e & 15) * 4) =
            make_uint2(f32x2_to_bf16x2(h4[0], h4[1]), f32x2_to_bf16x2(h4[2], h4[3]));
      }
    } else if (*s_last) {
      fence_acq_rel_gpu();
      const float4* all = reinterpret_cast<const float4*>(p.partials) + tile * S * P4;
      // two groups per thread per round, all S (<= 8) partials of both requested before any
      // is summed: the reduction costs one or two L2 round trips, not one per output
      for (int b = tid; b < n4; b += 2 * NTHR) {
        float4 x[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int e4 = b + u * NTHR;
#pragma unroll
          for (int qq = 0; qq < 8; ++qq)
            x[u][qq] = (qq < S && e4 < n4) ? __ldcg(all + qq * P4 + e4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int e4 = b + u * NTHR;
          if (e4 >= n4) continue;
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int qq = 0; qq < 8; ++qq)   // split order: deterministic
            if (qq < S) v = make_float4(v.x + x[u][qq].x, v.y + x[u][qq].y, v.z + x[u][qq].z, v.w + x[u][qq].w);
          const int tok = e4 >> 5;
          const int64_t n = row_tile * GV_ROWS + (e4 & 31) * 4;
          const float mul = ldexpf(st, pexp_s[tok]);
          uint16_t* dst = p.Y + (row_base + tok) * p.n_rows + n;
          const uint32_t lo = f32x2_to_bf16x2(v.x * mul, v.y * mul), hi = f32x2_to_bf16x2(v.z * mul, v.w * mul);
          if (n + 3 < p.n_rows && (p.n_rows & 3) == 0) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
          } else {
            const uint16_t o4[4] = {static_cast<uint16_t>(lo), static_cast<uint16_t>(lo >> 16),
                                    static_cast<uint16_t>(hi), static_cast<uint16_t>(hi >> 16)};
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (n + c < p.n_rows) dst[c] = o4[c];
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Gathered-row GEMV with argmax, row-streaming form (one 8-token n-tile).
// Candidate rows are random rows of the weight, so they are fetched whole:
// per stage, 16 candidates x full K, each row's codes and scales with one
// bulk copy each (a few large copies instead of many 128-byte tile gathers).
// The activation fragments of the whole K sit in shared memory for the
// kernel's lifetime. One persistent CTA per SM walks row groups b, b + G, ...
//   warps 0..7  consumers: warp w takes K-iterations [w n_it / 8, (w+1) n_it / 8)
//               of the stage's 16 rows; partial logits meet in a
//               double-buffered area, one named barrier per stage
//   warp 8      producer (lanes 0..15 copy one row's codes and scales each)
constexpr int RS_ROWS = 16;
constexpr int RS_STAGES = 2;
constexpr int RS_CONSUMERS = 8;
constexpr int RS_PRODUCER = RS_CONSUMERS;
constexpr int RS_THREADS = (RS_CONSUMERS + 1) * 32;

struct RsLayout {
  int code_stride, scale_stride, stage_bytes, x_bytes, smem;
};
// Row strides padded so that the 8 rows an MMA phase reads fall in distinct
// banks (code rows 64 bytes apart modulo 128).
inline RsLayout rs_layout(int64_t K) {
  RsLayout l;
  l.code_stride = static_cast<int>(K / 2 + 64);
  l.scale_stride = static_cast<int>(K / 16 + 16);
  l.stage_bytes = (RS_ROWS * (l.code_stride + l.scale_stride) + 127) / 128 * 128;
  l.x_bytes = static_cast<int>(K / GV_KIT) * 2048;
  l.smem = l.x_bytes + RS_STAGES * l.stage_bytes + 2 * RS_CONSUMERS * RS_ROWS * 8 * 4 + 1024 + 512;
  return l;
}

static __global__ void __launch_bounds__(RS_THREADS, 1)
    gather_rows_argmax_kernel(const TmaSkinnyParams p, RsLayout L) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t xs = base;
  const uint32_t ring = base + L.x_bytes;
  float* red = reinterpret_cast<float*>(base_ptr + L.x_bytes + RS_STAGES * L.stage_bytes);
  uint8_t* tail = base_ptr + L.x_bytes + RS_STAGES * L.stage_bytes + 2 * RS_CONSUMERS * RS_ROWS * 8 * 4;
  const uint32_t bar_base = smem_addr(tail);
  auto full_bar = [&](int q) { return bar_base + 8u * q; };
  auto empty_bar = [&](int q) { return bar_base + 8u * (RS_STAGES + q); };
  const uint32_t x_bar = bar_base + 8u * (2 * RS_STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + 64);
  int* s_last = reinterpret_cast<int*>(tail + 68);
  unsigned long long* kbest = reinterpret_cast<unsigned long long*>(tail + 128);   // [8]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int64_t KB = p.K / 2, KS = p.K / 16;
  const int n_it = static_cast<int>(p.K / GV_KIT);
  const int64_t n_groups = (p.n_rows + RS_ROWS - 1) / RS_ROWS;
  const int n_mine = static_cast<int>((n_groups - blockIdx.x + gridDim.x - 1) / gridDim.x);

  if (tid == 0) {
    for (int q = 0; q < RS_STAGES; ++q) {
      mbar_init(full_bar(q), 1);
      mbar_init(empty_bar(q), RS_CONSUMERS);
    }
    mbar_init(x_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < 8) kbest[tid] = 0ull;
  __syncthreads();

  if (warp == RS_PRODUCER) {
    // producer: lane r < 16 copies candidate row r of the group
    auto issue = [&](int i) {
      const int q = i % RS_STAGES;
      const uint32_t stage = ring + q * L.stage_bytes;
      const int64_t group = blockIdx.x + static_cast<int64_t>(i) * gridDim.x;
      if (lane == 0) mbar_arrive_expect_tx(full_bar(q), static_cast<uint32_t>(RS_ROWS * (KB + KS)));
      __syncwarp();
      if (lane < RS_ROWS) {
        const int64_t j0 = group * RS_ROWS + lane;
        const int64_t j = j0 < p.n_rows ? j0 : p.n_rows - 1;
        int64_t v = p.idx ? static_cast<int64_t>(p.idx[j]) : j;
        if (v < 0 || v >= p.w_rows) v = 0;   // a skipped entry reads row 0; its key is dropped
        bulk_load(stage + lane * L.code_stride, p.codes + v * KB, static_cast<uint32_t>(KB), full_bar(q));
        bulk_load(stage + RS_ROWS * L.code_stride + lane * L.scale_stride, p.scales + v * KS,
                  static_cast<uint32_t>(KS), full_bar(q));
      }
    };
    const int pre = n_mine < RS_STAGES ? n_mine : RS_STAGES;
    for (int i = 0; i < pre; ++i) issue(i);
    pdl_wait();   // the activation prep has finished and its writes are visible
    if (lane == 0) {
      mbar_arrive_expect_tx(x_bar, static_cast<uint32_t>(n_it) * 2048u);
      for (int it = 0; it < n_it; ++it)
        bulk_load(xs + it * 2048, p.xfrag + xfrag_unit(0, n_it, it, 0, 0, 0), 2048u, x_bar);
    }
    int issued = pre;
    for (int i = pre; i < n_mine; ++i) {
      const int q = i % RS_STAGES;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(empty_bar(q), ((i / RS_STAGES) - 1) & 1, abort_flag, p.status)))
        break;
      issue(i);
      ++issued;
    }
    // after a give-up, let the copies in flight land before the CTA exits
    if (lane == 0 && *abort_flag) {
      mbar_wait_bounded(x_bar, 0, nullptr, p.status, 100000000ull);
      const int first = issued > RS_STAGES ? issued - RS_STAGES : 0;
      for (int i = first; i < issued; ++i)
        mbar_wait_bounded(full_bar(i % RS_STAGES), (i / RS_STAGES) & 1, nullptr, p.status, 100000000ull);
    }
  } else {
    pdl_wait();   // the per-token shifts come from the prep
    const int it0 = warp * n_it / RS_CONSUMERS, it1 = (warp + 1) * n_it / RS_CONSUMERS;
    const float st = p.s_t[0];
    const int M = static_cast<int>(p.M);
    bool x_ready = false;
    for (int i = 0; i < n_mine; ++i) {
      const int q = i % RS_STAGES;
      float acc[1][1][4] = {{{0.f, 0.f, 0.f, 0.f}}};
      const bool ok = !*abort_flag && (x_ready || (x_ready = mbar_wait_bounded(x_bar, 0, abort_flag, p.status))) &&
                      mbar_wait_bounded(full_bar(q), (i / RS_STAGES) & 1, abort_flag, p.status);
      if (ok) {
        const uint32_t stage = ring + q * L.stage_bytes;
        const uint32_t rowA = stage + g * L.code_stride + t * 16;
        const uint32_t rowB = rowA + 8 * L.code_stride;
        const uint32_t scA0 = stage + RS_ROWS * L.code_stride + g * L.scale_stride + 2 * t;
        const uint32_t scB0 = scA0 + 8 * L.scale_stride;
        for (int it = it0; it < it1; ++it) {
          const uint4 ca = lds_v4(rowA + it * 64);
          const uint4 cb = lds_v4(rowB + it * 64);
          const uint32_t scA = e4m3x2_to_f16x2(lds_u16(scA0 + it * 8));
          const uint32_t scB = e4m3x2_to_f16x2(lds_u16(scB0 + it * 8));
          const uint32_t sa[2] = {dup_lo(scA), dup_hi(scA)}, sb[2] = {dup_lo(scB), dup_hi(scB)};
          const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w}, wb[4] = {cb.x, cb.y, cb.z, cb.w};
          const uint32_t xb = xs + it * 2048 + lane * 16;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint32_t fa[4], fb[4];
            e2m1x8_to_f16x2(wa[w], fa);
            e2m1x8_to_f16x2(wb[w], fb);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              fa[e] = hmul2(fa[e], sa[w >> 1]);
              fb[e] = hmul2(fb[e], sb[w >> 1]);
            }
            const uint32_t A0[4] = {fa[0], fb[0], fa[1], fb[1]}, A1[4] = {fa[2], fb[2], fa[3], fb[3]};
            const uint4 bx = lds_v4(xb + w * 512);
            mma_f16_16816(acc[0][0], A0, bx.x, bx.y);
            mma_f16_16816(acc[0][0], A1, bx.z, bx.w);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(q));
      }
      // partial logits of this warp: rows g, g + 8, tokens 2t, 2t + 1
      float* rb = red + (i & 1) * (RS_CONSUMERS * RS_ROWS * 8) + warp * (RS_ROWS * 8);
#pragma unroll
      for (int e = 0; e < 4; ++e) rb[(g + 8 * (e >> 1)) * 8 + 2 * t + (e & 1)] = acc[0][0][e];
      asm volatile("bar.sync 1, %0;" ::"r"(RS_CONSUMERS * 32) : "memory");
      if (tid < RS_ROWS * 8) {
        const int r = tid >> 3, tok = tid & 7;
        const int64_t j = (blockIdx.x + static_cast<int64_t>(i) * gridDim.x) * RS_ROWS + r;
        const int64_t vj = j < p.n_rows ? (p.idx ? static_cast<int64_t>(p.idx[j]) : j) : -1;
        if (tok < M && vj >= 0 && vj < p.w_rows) {
          const float* rr = red + (i & 1) * (RS_CONSUMERS * RS_ROWS * 8) + r * 8 + tok;
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < RS_CONSUMERS; ++w) v += rr[w * RS_ROWS * 8];
          const uint32_t vid = static_cast<uint32_t>(vj);
          atomicMax(&kbest[tok], (static_cast<unsigned long long>(float_order_key(v * ldexpf(st, p.pexp[tok])))
                                  << 32) | (0xFFFFFFFFu - vid));
        }
      }
    }
  }
  __syncthreads();
  // this CTA's per-token best into the global keys; the last CTA to finish
  // reads them out and leaves keys and counter at zero
  const int rows_in_chunk = static_cast<int>(p.M);
  if (tid < rows_in_chunk) atomicMax(&p.keys[tid], kbest[tid]);
  fence_acq_rel_gpu();
  __syncthreads();
  if (tid == 0) *s_last = atomicAdd(p.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (*s_last) {
    fence_acq_rel_gpu();
    for (int64_t m = tid; m < p.M; m += RS_THREADS) {
      const unsigned long long key = atomicExch(&p.keys[m], 0ull);
      p.out_ids[m] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
      if (p.out_logit) p.out_logit[m] = float_from_order_key(static_cast<uint32_t>(key >> 32));
    }
    if (tid == 0) atomicExch(p.counter, 0u);
  }
}

}  // namespace nvfp4
