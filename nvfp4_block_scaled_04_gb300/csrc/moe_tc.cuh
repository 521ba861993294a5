// Routed-expert GEMMs on the 5th-generation tensor cores, for layers whose
// experts receive many rows (MoE prefill: What 350+ Experiments Taught Us
// About Serving Qwen 3.6 35B-A3B, section 7, the NVFP4 mixture-of-experts
// kernel). Same arithmetic as the skinny expert kernel: the NVFP4 weight
// values e2m1 * e4m3 are exact in f16, the routed activations are f16 rows
// scaled by a power of two per row, products are exact and sums fp32.
//
// One CTA computes a tile of (expert, up to 128 of its routed rows, 128
// weight rows): D[w][t] = sum_k W[w][k] * X[t][k] with the weights as the A
// operand in tensor memory (M = 128) and the routed rows as the B operand in
// shared memory (N = the tile's rows rounded up to 32). Two CTAs share an SM
// (256 tensor-memory columns each), so one's prologue, pipeline fill and
// epilogue run beside the other's main loop. Measured at the 128-expert,
// top-8, H = 2048, I = 768 layer with 4096 tokens: 0.57 ms per layer against
// 0.69 ms with one CTA per SM on 256-row tiles and 0.61 ms with one CTA per
// SM computing 256 weight rows in two accumulators.
//   warp 0      TMA producer: each 64-K stage's weight codes (128 rows x 32 B)
//               and the tile's f16 rows (32-row boxes, 128B swizzle)
//   warp 1      tensor-memory allocation; lane 0 issues the MMAs
//               (tcgen05.mma.kind::f16, A from tensor memory)
//   warps 2..9  dequantise: warp w owns tensor-memory lanes 32 (w % 4).. and
//               one 32-K half of each stage, one weight row per thread: codes
//               -> f16 pairs (cvt e2m1x2), times the block scale (exact in
//               f16), tcgen05.st into the stage's A slot; then the epilogue
// Gate/up tiles hold 64 gate rows (lanes 0..63) and the matching 64 up rows
// (lanes 64..127); the epilogue stages both through shared memory, 32 routed
// rows at a time, and all eight warps write h = bf16(silu(g) * u). Down tiles
// write each routed row's expert output (bf16) for the combine kernel. The grid
// runs the weight blocks of one tile next to each other, so a tile's rows
// come from DRAM about once.
// Every mbarrier wait is bounded (device status word + CTA abort flag).
#pragma once

#include "tc_util.cuh"
#include "tcgen05.cuh"

namespace nvfp4 {
namespace {

constexpr int XT_BK = 64;                                // K per stage
constexpr int XT_NMAX = 128;                             // routed rows per tile
constexpr int XT_CTAS_PER_SM = 2;
constexpr int XT_STAGES = 4;                             // bounded by the A slots in tensor memory
constexpr int XT_B_BYTES = XT_NMAX * 128;                // rows x 64 f16
constexpr int XT_C_BYTES = 128 * 32;                     // 128 weight rows x 32 code bytes
constexpr int XT_STAGE_BYTES = XT_B_BYTES + XT_C_BYTES;  // a multiple of 1024
constexpr int XT_A_COL0 = XT_NMAX;                       // tensor memory: accumulator [0, NMAX), A slots after
constexpr int XT_TMEM_COLS = 256;                        // two CTAs per SM fill the 512 columns
constexpr int XT_DQ_WARPS = 8;
constexpr int XT_THREADS = (2 + XT_DQ_WARPS) * 32;
constexpr int XT_EPI_THREADS = XT_DQ_WARPS * 32;
constexpr int XT_BARS = 3 * XT_STAGES + 1;
constexpr int XT_SMEM = XT_STAGES * XT_STAGE_BYTES + 1024 /*alignment*/ + 256 /*barriers, slot, flag*/;
static_assert(XT_A_COL0 + XT_STAGES * 32 <= XT_TMEM_COLS, "tensor memory columns");
// a third CTA never fits an SM's 228 KB of shared memory, so the two
// resident CTAs' allocations never wait for each other
static_assert(3 * (XT_SMEM + 1024) > 228 * 1024 && XT_CTAS_PER_SM * XT_TMEM_COLS <= 512, "CTAs per SM");
static_assert(XT_BARS * 8 + 16 <= 256, "barrier area");
static_assert((2 * 64 * 33 + XT_NMAX) * 4 <= XT_STAGES * XT_STAGE_BYTES, "epilogue buffers fit in the ring");

struct MoeTcParams {
  const uint8_t* scales;   // row-major block scales of the stacked weights [E * rows_per_expert][K / 16]
  const float* s_t;        // per expert
  const int* pexp;         // per routed row: the power-of-two shift of its f16 copy
  const int* tile_count;
  const int* tile_expert;
  const int* tile_row0;
  const int* tile_rows;
  int K;                   // a multiple of 256
  int rows_per_expert;     // gate/up: 2I, down: H
  int inter;               // I
  int hidden;              // H
  uint16_t* h_out;         // gate/up: bf16 [routed rows][I]
  uint16_t* y_out;         // down: bf16 [routed rows][H]
  int* status;
};

// D (+)= A * B with A (M = 128, K = 16 f16) read from tensor memory.
NVFP4_DEV void tc_mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// AND of `pred` over the threads of the dequantising warps (named barrier 1).
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
__global__ void __launch_bounds__(XT_THREADS, XT_CTAS_PER_SM)
    moe_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                  const MoeTcParams p) {
  const int tile = static_cast<int>(blockIdx.y);
  if (tile >= *p.tile_count) return;
  const int wb = static_cast<int>(blockIdx.x);
  const int expert = p.tile_expert[tile];
  const int row0 = p.tile_row0[tile];
  const int nrows = p.tile_rows[tile];
  const int nbox = (nrows + 31) / 32;
  const int n_k = p.K / XT_BK;
  // first weight row of the tile in the stacked [E * rows_per_expert][K] matrix
  const int64_t wrow0 = static_cast<int64_t>(expert) * p.rows_per_expert + (GATEUP ? 64 * wb : 128 * wb);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bar_base = base + XT_STAGES * XT_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + XT_STAGES * XT_STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + XT_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + XT_BARS) + 1;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (XT_STAGES + s); };
  auto ready_bar = [&](int s) { return bar_base + 8u * (2 * XT_STAGES + s); };
  const uint32_t accf_bar = bar_base + 8u * (3 * XT_STAGES);
  auto stage_b = [&](int s) { return base + s * XT_STAGE_BYTES; };
  auto stage_c = [&](int s) { return base + s * XT_STAGE_BYTES + XT_B_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < XT_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(ready_bar(s), XT_DQ_WARPS);
    }
    mbar_init(accf_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_x) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_w) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(XT_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  int next_it = 0;   // producer: one past the last stage it issued
  if (warp == 0) {
    if (lane == 0) {
      for (int ks = 0; ks < n_k; ++ks) {
        const int s = ks % XT_STAGES;
        if (ks >= XT_STAGES &&
            !mbar_wait_bounded(empty_bar(s), ((ks / XT_STAGES) - 1) & 1, abort_flag, p.status))
          break;
        mbar_arrive_expect_tx(full_bar(s), XT_C_BYTES + static_cast<uint32_t>(nbox) * 4096u);
        if (GATEUP) {
          tma_load_2d(stage_c(s), &map_w, ks * 32, static_cast<int>(wrow0), full_bar(s));
          tma_load_2d(stage_c(s) + 2048, &map_w, ks * 32, static_cast<int>(wrow0 + p.inter), full_bar(s));
        } else {
          tma_load_2d(stage_c(s), &map_w, ks * 32, static_cast<int>(wrow0), full_bar(s));
        }
        for (int b = 0; b < nbox; ++b)
          tma_load_2d(stage_b(s) + 4096 * b, &map_x, ks * XT_BK, row0 + 32 * b, full_bar(s));
        next_it = ks + 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // kind::f16: f16 A and B, fp32 D, both K-major; N >> 3 at bit 17, M >> 4 at bit 24
      const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(nbox * 32 >> 3) << 17) | (uint32_t(128 >> 4) << 24);
      for (int ks = 0; ks < n_k; ++ks) {
        const int s = ks % XT_STAGES;
        // the dequantising warps arrive only after the stage's copies landed
        if (!mbar_wait_bounded(ready_bar(s), (ks / XT_STAGES) & 1, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < XT_BK / 16; ++k)
          tc_mma_f16_tmem_a(tmem, tmem + XT_A_COL0 + s * 32 + 8 * k, smem_desc(stage_b(s) + 32 * k, 16, 1024, 2),
                            idesc, (ks > 0 || k > 0) ? 1u : 0u);
        tc_commit(empty_bar(s));
      }
      // also after a give-up: the epilogue and the unwind wait for the MMAs issued so far
      tc_commit(accf_bar);
    }
  } else {
    const int dw = warp - 2;              // 0..7
    const int quarter = warp & 3;         // tensor-memory lane quarter
    const int half = dw >> 2;             // which 32 K of each stage
    const int r = quarter * 32 + lane;    // tensor-memory lane = weight row of the tile
    const int64_t grow = GATEUP ? (r < 64 ? wrow0 + r : wrow0 + p.inter + (r - 64)) : wrow0 + r;
    const uint32_t a_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + XT_A_COL0 + 16 * half;
    // block scales: 16 bytes of a row cover four stages (K % 256 == 0), word j
    // the four 16-K blocks of stage j; group g + 1 is requested while group g
    // is in use
    const uint4* sgrp = reinterpret_cast<const uint4*>(p.scales + grow * (p.K / 16));
    const int n_grp = n_k / 4;
    uint4 sc_cur = __ldg(sgrp), sc_next = n_grp > 1 ? __ldg(sgrp + 1) : make_uint4(0u, 0u, 0u, 0u);
    bool ok = true;
    for (int ks = 0; ks < n_k; ++ks) {
      const int s = ks % XT_STAGES;
      if ((ks & 3) == 0 && ks > 0) {
        sc_cur = sc_next;
        if ((ks >> 2) + 1 < n_grp) sc_next = __ldg(sgrp + (ks >> 2) + 1);
      }
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(full_bar(s), (ks / XT_STAGES) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      const uint32_t sc = (ks & 3) == 0 ? sc_cur.x : (ks & 3) == 1 ? sc_cur.y : (ks & 3) == 2 ? sc_cur.z : sc_cur.w;
      const uint32_t s01 = e4m3x2_to_f16x2(half ? (sc >> 16) : (sc & 0xFFFFu));
      const uint32_t bscale[2] = {dup_lo(s01), dup_hi(s01)};
      const uint4 c = lds128(stage_c(s) + r * 32 + 16 * half);
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t f[4];
        e2m1x8_to_f16x2(w[j], f);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[4 * j + i] = hmul2(f[i], bscale[j / 2]);
      }
      tc_st_16cols(a_lane + s * 32, v);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ready_bar(s));
    }

    // epilogue: every warp takes part in the named barriers whatever happened above
    const bool acc_ok = __all_sync(0xffffffffu, mbar_wait_bounded(accf_bar, 0, abort_flag, p.status));
    tc_fence_after();
    if (xt_all_epilogue(ok && acc_ok && *abort_flag == 0)) {
      // the ring is free once the MMAs completed: gate and up values of 32
      // routed rows ([64][33] each, padded against bank conflicts), then the
      // per-row output multipliers s_t * 2^shift
      float* gbuf = reinterpret_cast<float*>(base_ptr);
      float* ubuf = gbuf + 64 * 33;
      float* mulv = ubuf + 64 * 33;
      const float st = p.s_t[expert];
      const int et = threadIdx.x - 64;
      if (et < nrows) mulv[et] = ldexpf(st, p.pexp[row0 + et]);
      xt_epilogue_sync();
      for (int j = 0; j < nbox; ++j) {
        uint32_t acc[16];
        tc_ld_16cols(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(32 * j + 16 * half),
                     acc);
        tc_wait_ld();
        if (GATEUP) {
          float* dst = (quarter < 2 ? gbuf : ubuf) + (32 * (quarter & 1) + lane) * 33 + 16 * half;
#pragma unroll
          for (int i = 0; i < 16; ++i) dst[i] = __uint_as_float(acc[i]);
          xt_epilogue_sync();
          // thread: intermediate row n = lane + 32 (dw & 1), routed rows 8 (dw >> 1) .. + 8
          const int n = lane + 32 * (dw & 1), c0 = 8 * (dw >> 1);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int t = 32 * j + c0 + i;
            if (t < nrows) {
              const float m = mulv[t];
              const float g = gbuf[n * 33 + c0 + i] * m;
              const float u = ubuf[n * 33 + c0 + i] * m;
              const float h = g / (1.0f + expf(-g)) * u;
              p.h_out[static_cast<int64_t>(row0 + t) * p.inter + 64 * wb + n] =
                  static_cast<uint16_t>(f32_to_bf16_bits(h));
            }
          }
          xt_epilogue_sync();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int t = 32 * j + 16 * half + i;
            if (t < nrows)
              p.y_out[static_cast<int64_t>(row0 + t) * p.hidden + 128 * wb + r] =
                  static_cast<uint16_t>(f32_to_bf16_bits(__uint_as_float(acc[i]) * mulv[t]));
          }
        }
      }
    }
  }

  // Unwind: after a give-up, copies and MMAs already issued land (bounded)
  // before the shared and tensor memory they target go away.
  if (warp == 0 && lane == 0 && *abort_flag) {
    for (int it = next_it - 1; it >= 0 && it >= next_it - XT_STAGES; --it)
      mbar_wait_bounded(full_bar(it % XT_STAGES), (it / XT_STAGES) & 1, nullptr, p.status, 100000000ull);
  }
  if (warp == 1 && lane == 0 && *abort_flag) mbar_wait_bounded(accf_bar, 0, nullptr, p.status, 100000000ull);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(XT_TMEM_COLS) : "memory");
  }
}

}  // namespace
}  // namespace nvfp4
