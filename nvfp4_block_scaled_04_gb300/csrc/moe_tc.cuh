// Routed-expert GEMMs on the 5th-generation tensor cores, for layers whose
// experts receive many rows (MoE prefill: What 350+ Experiments Taught Us
// About Serving Qwen 3.6 35B-A3B, section 7, the NVFP4 mixture-of-experts
// kernel). Same arithmetic as the skinny expert kernel: the NVFP4 weight
// values e2m1 * e4m3 are exact in f16, the routed activations are f16 rows
// scaled by a power of two per row, products are exact and sums fp32.
//
// A work item is (tile, pair of weight blocks): up to 256 routed rows of one
// expert against 2 x 128 weight rows, D[w][t] = sum_k W[w][k] * X[t][k]. Two
// CTAs of a cluster share an item: each dequantises its own 128 weight rows
// into its tensor memory (the A operand) and loads one half of the tile's
// routed rows (the B operand, f16, 128B swizzle), and one thread of the even
// CTA issues tcgen05.mma.cta_group::2.kind::f16 (M = 256, N = the tile's rows
// rounded up to 32), which accumulates each CTA's 128 rows into that CTA's
// tensor memory. The kernel is persistent: pair i walks items i, i + pairs,
// ... (the weight blocks of one tile next to each other, so a tile's rows
// come from L2), and the stage ring runs on across items.
//
// Cost model (measured on this layer): the weights of an item are converted
// once whatever its N, and the conversion of a 64-K step (~345 clocks per SM
// for 128 rows) is slower than its MMAs at N = 128 (256 clocks), so tiles
// take up to 256 routed rows (512 clocks of MMAs per step) and the routing
// plan splits an expert's rows into equal tiles. The TMA engine's rate of
// row requests also bounds the ring, so the weight codes arrive as 64-byte
// rows (two 64-K steps per request, 64B swizzle so the dequantising warps'
// 16-byte reads of 32 rows hit distinct banks) and the routed rows as 128-row
// boxes of 128-byte rows.
//   warps 0, 26   TMA producers, taking alternate 128-K stages
//   warp 1        tensor-memory allocation; in the even CTA lane 0 issues
//                 the MMAs (A from tensor memory)
//   warps 2..9    dequantise, in two groups of four that take the first and
//                 the second 64-K step of each stage: warp w owns tensor-memory
//                 lanes 32 (w % 4).., one weight row per thread: codes -> f16
//                 pairs (cvt e2m1x2), times the block scale (exact in f16),
//                 tcgen05.st into the step's A slot (stage s, step q: slot 2 s + q)
//   warps 10..25  epilogue: warp w reads tensor-memory lanes 32 (w % 4).. of
//                 every fourth 32-column group of the accumulator
// Gate/up blocks interleave their rows: tensor-memory lane 2n holds gate row
// n of the block and lane 2n + 1 up row n, so one shfl.xor gives each thread
// both values and h = bf16(silu(g) * u) needs no shared-memory exchange. The
// accumulator (256 columns) leaves no room for a second one, so the MMAs of
// the next item wait until every epilogue warp has read its last column group
// (measured with wait counters: the MMA thread spent 29% (gate/up) and 48%
// (down) of its time there while the epilogue wrote 2-byte scattered
// stores). So the epilogue stages each warp's 32 routed rows in shared memory
// and writes them with one TMA store, and sixteen epilogue warps (each with
// at most two column groups) release the accumulator after at most one group
// of work; the dequantising warps were idle two thirds of the time, so eight
// of them do that work.
// Down blocks write each routed row's expert output (bf16) for the combine
// kernel.
//
// Synchronisation, per CTA unless stated:
//   full[s]     this CTA's codes and routed rows of stage s landed
//   empty[s]    the pair's MMAs have consumed stage s and its two A slots
//               (one multicast commit); the producer and the dequantising
//               warps wait on it before reusing them
//   ready[s]    in the even CTA only: both CTAs' dequantising warps have
//               filled stage s's A slots (16 arrivals, 8 remote)
// The MMA thread waits once and commits once per stage (eight MMAs): a wait,
// a fence and a commit around every four MMAs cost about as much issue time
// as the MMAs of a 128-row tile take (measured on a probe).
//   accf        the accumulator holds a finished item (one multicast commit)
//   acce        in the even CTA only: both CTAs' epilogues have read the
//               accumulator (32 arrivals, 16 remote)
// Every wait is bounded (device status word + CTA abort flag), and both CTAs
// reach the closing cluster barrier on every path, so a CTA never leaves
// while its peer may still touch its memory.
#pragma once

#include "tc_util.cuh"
#include "tcgen05.cuh"

namespace nvfp4 {
namespace {

constexpr int XT_BK = 64;                                // K per step (one A slot)
constexpr int XT_SUB = 2;                                // steps per stage
constexpr int XT_NMAX = 256;                             // routed rows per tile
constexpr int XT_STAGES = 4;                             // shared-memory ring
constexpr int XT_ASLOTS = 2 * XT_STAGES;                 // A slots in tensor memory: two per stage
constexpr int XT_B_SUB = XT_NMAX / 2 * 128;              // this CTA's half of the rows x 64 f16
constexpr int XT_B_BYTES = XT_SUB * XT_B_SUB;
constexpr int XT_C_BYTES = 128 * 64;                     // 128 weight rows x 64 code bytes (128 K)
constexpr int XT_STAGE_BYTES = XT_B_BYTES + XT_C_BYTES;  // a multiple of 1024
constexpr int XT_A_COL0 = XT_NMAX;                       // tensor memory: the accumulator, then the A slots
constexpr int XT_TMEM_COLS = 512;
constexpr int XT_DQ_GROUP = 4;                           // warps converting one step in one CTA
constexpr int XT_DQ_WARPS = 2 * XT_DQ_GROUP;
constexpr int XT_DQ_WARP0 = 2;
constexpr int XT_EPI_WARPS = 16;
constexpr int XT_EPI_WARP0 = XT_DQ_WARP0 + XT_DQ_WARPS;
constexpr int XT_PROD1_WARP = XT_EPI_WARP0 + XT_EPI_WARPS;   // the second producer
constexpr int XT_THREADS = (XT_PROD1_WARP + 1) * 32;
constexpr int XT_EPI_THREADS = XT_EPI_WARPS * 32;
// full[S], empty[S], ready[S], accumulator full / empty, MMA drain
constexpr int XT_BARS = 3 * XT_STAGES + 3;
// output staging: per epilogue warp two buffers of 32 routed rows x 32 bf16
// (gate/up uses 16 of the 32 columns); per-row multipliers
constexpr int XT_STG_BYTES = 32 * 64;
constexpr int XT_EPI_BYTES = XT_EPI_WARPS * 2 * XT_STG_BYTES + XT_NMAX * 4;
constexpr int XT_SMEM = XT_STAGES * XT_STAGE_BYTES + XT_EPI_BYTES + 1024 /*alignment*/ + 256 /*barriers, slot, flag*/;
static_assert(XT_A_COL0 + XT_ASLOTS * 32 <= XT_TMEM_COLS, "tensor memory columns");
static_assert(XT_SUB == 2 && XT_ASLOTS == XT_SUB * XT_STAGES, "the two dequant groups take the two steps of a stage");
// a second CTA never fits an SM's 228 KB of shared memory (nor its registers),
// so the CTA's allocation of all 512 tensor-memory columns never waits
static_assert(2 * (XT_SMEM + 1024) > 228 * 1024, "one CTA per SM");
static_assert(XT_BARS * 8 + 16 <= 256, "barrier area");
static_assert(XT_NMAX / 32 <= 2 * 4, "at most two 32-column groups per epilogue warp (four warps per lane quarter)");

struct MoeTcParams {
  const uint8_t* scales;   // row-major block scales of the stacked weights [E * rows_per_expert][K / 16]
  const float* s_t;        // per expert
  const int* pexp;         // per routed row: the power-of-two shift of its f16 copy
  const int* tile_count;
  const int* tile_expert;
  const int* tile_row0;
  const int* tile_rows;    // 1 .. XT_NMAX
  int K;                   // a multiple of 256
  int rows_per_expert;     // gate/up: 2I, down: H
  int inter;               // I (a multiple of 256)
  int hidden;              // H (a multiple of 256)
  uint16_t* h_out;         // gate/up: bf16 [routed rows][I]
  uint16_t* y_out;         // down: bf16 [routed rows][H]
  int* status;
};

// D (+)= A * B over the CTA pair (M = 256), A (K = 16 f16) read from each
// CTA's tensor memory, B from each CTA's shared memory (one half of N each).
NVFP4_DEV void tc_mma_f16_tmem_a_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// AND of `pred` over the epilogue warps (named barrier 1).
NVFP4_DEV bool xt_all_epilogue(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(pred)), "n"(XT_EPI_THREADS)
      : "memory");
  return out != 0;
}
NVFP4_DEV void xt_epilogue_sync() { asm volatile("bar.sync 1, %0;" ::"n"(XT_EPI_THREADS) : "memory"); }

template <bool GATEUP>
__global__ void __launch_bounds__(XT_THREADS, 1)
    moe_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                  const __grid_constant__ CUtensorMap map_out, const MoeTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t stg_base = base + XT_STAGES * XT_STAGE_BYTES;                      // 1024-aligned
  float* mulv = reinterpret_cast<float*>(base_ptr + XT_STAGES * XT_STAGE_BYTES + XT_EPI_WARPS * 2 * XT_STG_BYTES);
  const uint32_t bar_base = base + XT_STAGES * XT_STAGE_BYTES + XT_EPI_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + XT_STAGES * XT_STAGE_BYTES + XT_EPI_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + XT_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + XT_BARS) + 1;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (XT_STAGES + s); };
  auto ready_bar = [&](int s) { return bar_base + 8u * (2 * XT_STAGES + s); };
  const uint32_t accf_bar = bar_base + 8u * (3 * XT_STAGES);
  const uint32_t acce_bar = accf_bar + 8u;
  const uint32_t drain_bar = accf_bar + 16u;
  auto stage_b = [&](int s) { return base + s * XT_STAGE_BYTES; };
  auto stage_c = [&](int s) { return base + s * XT_STAGE_BYTES + XT_B_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair_id = static_cast<int>(blockIdx.x >> 1), n_pairs = static_cast<int>(gridDim.x >> 1);
  const int n_bpairs = (GATEUP ? p.inter / 64 : p.hidden / 128) / 2;
  const int n_work = *p.tile_count * n_bpairs;
  const int n_st = p.K / (XT_SUB * XT_BK);   // stages per item (even)
  if (threadIdx.x == 0) {
    for (int s = 0; s < XT_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(ready_bar(s), 2 * XT_DQ_WARPS);
    }
    mbar_init(accf_bar, 1);
    mbar_init(acce_bar, 2 * XT_EPI_WARPS);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_x) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_w) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_out) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(XT_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();   // both CTAs' barriers and tensor memory exist before anything refers to them
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  int next_it = 0;   // producer: one past the last stage it issued
  const int prod = warp == 0 ? 0 : (warp == XT_PROD1_WARP ? 1 : -1);
  if (prod >= 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int w = pair_id; w < n_work && ok; w += n_pairs) {
        const int t = w / n_bpairs, wb = 2 * (w - t * n_bpairs) + static_cast<int>(rank);
        const int expert = p.tile_expert[t], nbox = (p.tile_rows[t] + 31) / 32;
        // this CTA's half of the tile's (32 nbox) rows starts here; the box
        // is 128 rows whatever the tile holds (rows past the half are unused)
        const int brow0 = p.tile_row0[t] + static_cast<int>(rank) * 16 * nbox;
        const int wrow0 = expert * p.rows_per_expert + (GATEUP ? 64 * wb : 128 * wb);
        for (int ks = 0; ks < n_st; ++ks, ++it) {
          if ((it & 1) != prod) continue;
          const int s = it % XT_STAGES;
          if (it >= XT_STAGES &&
              !mbar_wait_cluster_bounded(empty_bar(s), ((it / XT_STAGES) - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), XT_C_BYTES + XT_B_BYTES);
          if (GATEUP)
            tma_load_3d(stage_c(s), &map_w, ks * 64, wrow0, 0, full_bar(s));   // gate rows, then up rows
          else
            tma_load_2d(stage_c(s), &map_w, ks * 64, wrow0, full_bar(s));
#pragma unroll
          for (int q = 0; q < XT_SUB; ++q)
            tma_load_2d(stage_b(s) + q * XT_B_SUB, &map_x, (XT_SUB * ks + q) * XT_BK, brow0, full_bar(s));
          next_it = it + 1;
        }
      }
    }
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      int it = 0, item = 0;
      bool ok = true;
      for (int w = pair_id; w < n_work && ok; w += n_pairs, ++item) {
        // both CTAs' epilogues have read the accumulator's previous item
        if (item > 0 && !mbar_wait_cluster_bounded(acce_bar, (item - 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const int t = w / n_bpairs;
        const int nbox = (p.tile_rows[t] + 31) / 32;
        // kind::f16: f16 A and B, fp32 D, both K-major; N >> 3 at bit 17, M >> 4 at bit 24
        const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(nbox * 32 >> 3) << 17) | (uint32_t(256 >> 4) << 24);
        for (int ks = 0; ks < n_st; ++ks, ++it) {
          const int s = it % XT_STAGES;
          // the dequantising warps of both CTAs arrive only after their stage's copies landed
          if (!mbar_wait_cluster_bounded(ready_bar(s), (it / XT_STAGES) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = tmem + XT_A_COL0 + static_cast<uint32_t>(s) * (XT_SUB * 32);
          const uint64_t b0 = smem_desc(stage_b(s), 16, 1024, 2);
#pragma unroll
          for (int q = 0; q < XT_SUB; ++q)
#pragma unroll
            for (int k = 0; k < XT_BK / 16; ++k)
              // A: 8 columns per 16 K; B: the descriptor's address field counts 16 bytes
              tc_mma_f16_tmem_a_pair(tmem, a0 + 32 * q + 8 * k, b0 + static_cast<uint64_t>((q * XT_B_SUB + 32 * k) >> 4),
                                     idesc, (ks > 0 || q > 0 || k > 0) ? 1u : 0u);
          tc_commit_pair(empty_bar(s));
        }
        if (ok) tc_commit_pair(accf_bar);
      }
      // every MMA issued so far has completed before either CTA frees its memory
      tc_commit_pair(drain_bar);
      mbar_wait_cluster_bounded(drain_bar, 0, nullptr, p.status);
    }
  } else if (warp >= XT_DQ_WARP0 && warp < XT_EPI_WARP0) {
    const int dw = warp - XT_DQ_WARP0;                 // 0..7
    const int grp = dw / XT_DQ_GROUP;                  // the step of each stage this warp converts
    const int quarter = warp & 3;                      // tensor-memory lane quarter
    const int r = quarter * 32 + lane;                 // tensor-memory lane
    // its weight row: down r; gate/up gate row r / 2 (r even) or up row r / 2
    // (r odd), which the codes box holds at row r / 2, resp. 64 + r / 2
    const int crow = GATEUP ? ((r & 1) ? 64 + (r >> 1) : (r >> 1)) : r;
    const uint32_t a_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + XT_A_COL0;
    int it0 = 0;                                       // the item's first stage
    bool ok = true;
    for (int w = pair_id; w < n_work && ok; w += n_pairs, it0 += n_st) {
      const int t = w / n_bpairs, wb = 2 * (w - t * n_bpairs) + static_cast<int>(rank);
      const int64_t wrow0 = static_cast<int64_t>(p.tile_expert[t]) * p.rows_per_expert + (GATEUP ? 64 * wb : 128 * wb);
      const int64_t grow = GATEUP ? ((r & 1) ? wrow0 + p.inter + (r >> 1) : wrow0 + (r >> 1)) : wrow0 + r;
      // block scales: 16 bytes of a row cover two stages (word 2 (ks % 2) + q:
      // the four 16-K blocks of step q of stage ks); the next pair of stages'
      // are requested one ahead
      const uint4* sgrp = reinterpret_cast<const uint4*>(p.scales + grow * (p.K / 16));
      uint4 sc_cur = make_uint4(0u, 0u, 0u, 0u), sc_next = __ldg(sgrp);
      for (int ks = 0; ks < n_st && ok; ++ks) {
        if ((ks & 1) == 0) {
          sc_cur = sc_next;
          if (ks / 2 + 1 < n_st / 2) sc_next = __ldg(sgrp + ks / 2 + 1);
        }
        const int it = it0 + ks, s = it % XT_STAGES;
        const int a = XT_SUB * s + grp;               // this step's A slot
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(full_bar(s), (it / XT_STAGES) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        // the A slot is free once the MMAs of stage it - XT_STAGES completed
        if (it >= XT_STAGES &&
            !__all_sync(0xffffffffu, mbar_wait_cluster_bounded(empty_bar(s), ((it / XT_STAGES) - 1) & 1, abort_flag,
                                                               p.status))) {
          ok = false;
          break;
        }
        const uint32_t sc = (ks & 1) == 0 ? (grp ? sc_cur.y : sc_cur.x) : (grp ? sc_cur.w : sc_cur.z);
        // the row's 32 code bytes of this step: 16-byte chunks 2 grp, 2 grp + 1
        // at their 64B-swizzled places
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t s01 = e4m3x2_to_f16x2(hf ? (sc >> 16) : (sc & 0xFFFFu));
          const uint32_t bscale[2] = {dup_lo(s01), dup_hi(s01)};
          const int c16 = 2 * grp + hf;
          const uint4 c = lds128(stage_c(s) + crow * 64 + ((c16 ^ ((crow >> 1) & 3)) << 4));
          const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
          uint32_t v[16];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t f[4];
            e2m1x8_to_f16x2(wv[e], f);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[4 * e + i] = hmul2(f[i], bscale[e / 2]);
          }
          tc_st_16cols(a_lane + a * 32 + 16 * hf, v);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(ready_bar(s), 0);
      }
    }
  } else if (warp >= XT_EPI_WARP0 && warp < XT_EPI_WARP0 + XT_EPI_WARPS) {
    // epilogue: every epilogue warp takes part in the named barrier of an
    // item; a failed wait is agreed on by all sixteen (bar.red) before any leaves
    const int quarter = warp & 3;
    const int ew = warp - XT_EPI_WARP0;               // 0..15
    const int ch = ew >> 2;                           // column groups j with j % 4 == ch
    const int et = threadIdx.x - XT_EPI_WARP0 * 32;   // 0..511
    const uint32_t lanes = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t stg = stg_base + static_cast<uint32_t>(ew) * 2 * XT_STG_BYTES;
    // output columns of this warp within the block: gate/up 16 intermediate
    // columns (lane pair 2n, 2n + 1 -> column n), down 32 columns
    constexpr int OCOLS = GATEUP ? 16 : 32;
    int item = 0, nstore = 0;
    for (int w = pair_id; w < n_work; w += n_pairs, ++item) {
      const int t = w / n_bpairs, wb = 2 * (w - t * n_bpairs) + static_cast<int>(rank);
      const int expert = p.tile_expert[t], row0 = p.tile_row0[t], nrows = p.tile_rows[t];
      const int nbox = (nrows + 31) / 32;
      const int col0 = GATEUP ? 64 * wb + 16 * quarter : 128 * wb + 32 * quarter;
      xt_epilogue_sync();   // the previous item's reads of mulv are done
      const float st = p.s_t[expert];
      if (et < nrows) mulv[et] = ldexpf(st, p.pexp[row0 + et]);
      const bool got = __all_sync(0xffffffffu, mbar_wait_cluster_bounded(accf_bar, item & 1, abort_flag, p.status));
      if (!xt_all_epilogue(got && *abort_flag == 0)) break;
      tc_fence_after();
      // phase A: read this warp's column groups (at most two: j = ch, ch + 4)
      // and form their outputs as bf16 pairs in registers, then release the
      // accumulator; phase B stages and stores them. (Staging and storing a
      // group before reading the next held the next item's MMAs: the MMA
      // thread waited for the epilogue 16% / 30% of its time.)
      constexpr int OW = GATEUP ? 8 : 16;   // output words of a group per thread
      uint32_t ob[2][OW];
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2) {
        const int j = ch + 4 * g2;
        if (j >= nbox) continue;
        if (GATEUP) {
          uint32_t a[32];
          tc_ld_32cols(tmem + lanes + static_cast<uint32_t>(32 * j), a);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            // even lane (gate): routed row 2i; odd lane (up): routed row 2i + 1
            const uint32_t mine = (lane & 1) ? a[2 * i + 1] : a[2 * i];
            const uint32_t give = (lane & 1) ? a[2 * i] : a[2 * i + 1];
            const uint32_t other = __shfl_xor_sync(0xffffffffu, give, 1);
            const int c = 2 * i + (lane & 1);
            const float m = mulv[32 * j + c];
            const float g = __uint_as_float((lane & 1) ? other : mine) * m;
            const float u = __uint_as_float((lane & 1) ? mine : other) * m;
            const uint32_t h = f32_to_bf16_bits(__fdividef(g, 1.0f + __expf(-g)) * u);
            ob[g2][i >> 1] = (i & 1) ? (ob[g2][i >> 1] | (h << 16)) : h;
          }
        } else {
          // in 16-column halves (registers)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t a[16];
            tc_ld_16cols(tmem + lanes + static_cast<uint32_t>(32 * j + 16 * hh), a);
            tc_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; c += 2)
              ob[g2][8 * hh + (c >> 1)] = f32x2_to_bf16x2(__uint_as_float(a[c]) * mulv[32 * j + 16 * hh + c],
                                                          __uint_as_float(a[c + 1]) * mulv[32 * j + 16 * hh + c + 1]);
          }
        }
      }
      // the accumulator's last reads of this item: let the MMAs of the next one start
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_bar, 0);
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2) {
        const int j = ch + 4 * g2;
        if (j >= nbox) continue;
        // this warp's staging buffer: the tensor store that last read it is done
        const uint32_t buf = stg + static_cast<uint32_t>(nstore & 1) * XT_STG_BYTES;
        ++nstore;
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncwarp();
        // staging layout: routed row c of the group at buf + c * 2 OCOLS, bf16 columns
        if (GATEUP) {
          const int n = lane >> 1;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = 2 * i + (lane & 1);
            const uint16_t h = static_cast<uint16_t>(ob[g2][i >> 1] >> (16 * (i & 1)));
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(buf + c * (2 * OCOLS) + 2 * n), "h"(h) : "memory");
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const uint16_t y = static_cast<uint16_t>(ob[g2][c >> 1] >> (16 * (c & 1)));
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(buf + c * (2 * OCOLS) + 2 * lane), "h"(y) : "memory");
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the tensor store
        __syncwarp();
        if (32 * j + 32 <= nrows) {
          if (lane == 0) {
            asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(&map_out),
                         "r"(col0), "r"(row0 + 32 * j), "r"(buf)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        } else {
          // the tile's ragged last rows: a box would write into the next tile
          const int c = lane;
          if (32 * j + c < nrows) {
            uint16_t* dst = (GATEUP ? p.h_out : p.y_out) +
                            static_cast<int64_t>(row0 + 32 * j + c) * (GATEUP ? p.inter : p.hidden) + col0;
#pragma unroll
            for (int q = 0; q < OCOLS / 8; ++q)
              reinterpret_cast<uint4*>(dst)[q] = lds128(buf + c * (2 * OCOLS) + 16 * q);
          }
        }
      }
    }
    // stores complete before the CTA exits
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }

  // Unwind after a give-up: copies already issued land (bounded) before the
  // shared memory they target goes away; the MMA thread drained its MMAs above.
  if (prod >= 0 && lane == 0 && *abort_flag) {
    for (int it = next_it - 1; it >= 0 && it >= next_it - XT_STAGES; --it)
      if ((it & 1) == prod)
        mbar_wait_bounded(full_bar(it % XT_STAGES), (it / XT_STAGES) & 1, nullptr, p.status, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // the peer is done with this CTA's shared and tensor memory
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(XT_TMEM_COLS) : "memory");
  }
}

}  // namespace
}  // namespace nvfp4
