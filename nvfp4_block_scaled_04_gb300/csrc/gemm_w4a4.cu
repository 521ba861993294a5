// W4A4 NVFP4 GEMM on the 5th-generation tensor cores (sm_103a):
//   Y[m][n] = bf16( s_tA * s_tW * sum_k a[m][k] * w[n][k] )
// with a, w the e2m1 * e4m3 block-scaled values: both operands 4-bit, run
// natively on Blackwell (52.6% More Tokens, 1.53x Less GPU Time: Production
// Inference with Minima and Rafay, comparison paragraph). The block-scaled MMA multiplies the e2m1 codes and
// the per-16 E4M3 scales and accumulates in fp32 in tensor memory; the
// epilogue applies the two fp32 tensor scales and rounds to bf16.
//
// A persistent CTA per SM computes 128 x 256 output tiles. Each stage of a
// 4-deep shared-memory ring holds 256 K of the A and W code tiles (128B
// swizzle) and their block scales, already in the MMA scale layout (one
// 512-byte atom per 128 rows x 64 K).
//
// The block scales reach tensor memory through registers: four scale warps,
// one per tensor-memory lane quarter, read each stage's atoms from shared
// memory and write them with tcgen05.st. Copying them with tcgen05.cp costs
// about as much tensor-pipe time per instruction as a 128 x 256 x 64 MMA
// (measured on sm_103a: ~100 vs ~128 clocks), and one stage needs twelve
// atoms, so on the tensor pipe the copies took longer than the MMAs they
// fed; tcgen05.st from other warps runs beside the MMAs without slowing them.
// Every mbarrier wait is bounded; a wait that gives up records
// NVFP4_ERR_TIMEOUT in a device status word and the CTA unwinds, frees its
// tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "quant_core.cuh"
#include "tc_util.cuh"
#include "tcgen05.cuh"

namespace nvfp4 {

__device__ int g_device_status = 0;

int* device_status_ptr() {
  static int* cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(p);
  }
  return cached[dev];
}

namespace {

// Tile: 128 rows of A x 256 rows of W per MMA tile, 256 K-elements per stage.
constexpr int BM = 128, BN = 256;
constexpr int BK = 256;                     // K elements per stage (128 bytes of codes per row)
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 8;                // two per TMEM lane quarter, one per 128-column half
constexpr int EPI_WARP0 = 3;                // warps 0, 2 produce (even / odd stages), warp 1 issues MMAs
constexpr int SF_WARPS = 4;                 // one per TMEM lane quarter
constexpr int SF_WARP0 = EPI_WARP0 + EPI_WARPS;
constexpr int THREADS = (SF_WARP0 + SF_WARPS) * 32;
constexpr int A_BYTES = BM * 128;           // 16 KB
constexpr int B_BYTES = BN * 128;           // 32 KB
constexpr int SFA_BYTES = 4 * 512;          // 4 scale atoms (128 rows x 64 K each)
constexpr int SFB_BYTES = 2 * 4 * 512;      // 2 row halves x 4 atoms
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;   // 54 KB
constexpr int TMEM_COLS = 512;              // 256 accumulator + 4 stages x (16 + 32) scale columns
constexpr int SF_TMEM_BASE = 256;
constexpr int SF_COLS_PER_STAGE = 48;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
static_assert((3 * STAGES + 4) * 8 <= 256, "barrier area");
constexpr int BAND = 32;                    // m-tiles that share one sweep over the W tiles

// Instruction descriptor: kind::mxf4nvf4, A and B E2M1 (1), both K-major,
// N>>3 at bit 17, UE4M3 scales (bit 23 = 0), M>>4 at bit 24.
constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

NVFP4_DEV void tc_mma_mxf4nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                               uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}


struct W4A4Params {
  const uint8_t* sfa;   // MMA-layout scales of A
  const uint8_t* sfb;   // MMA-layout scales of W
  const float* st_a;
  const float* st_b;
  uint16_t* Y;
  int M, N, K;
  int m_tiles, n_tiles;
  // EPI_QUANT: the output as NVFP4 with tensor scale *q_st (N % 64 == 0)
  uint8_t* q_codes;          // [M][N/2]
  uint8_t* q_scales;         // MMA layout: rows padded to 128, N/16 scale columns
  const float* q_st;
  // EPI_AMAX: max |bf16 output| as fp32 bits (atomicMax; zero on entry)
  unsigned int* amax_bits;
};

// What an epilogue thread does with its row's 128 bf16 outputs (packed in
// pairs: packed[i] holds columns 2i, 2i + 1):
//   EPI_BF16   store them (Y)
//   EPI_QUANT  quantise them to NVFP4 with the given tensor scale (the same
//              per-16 block step as the quantiser, on the bf16 values the
//              unfused layer would hand on) and store codes and MMA-layout
//              scales; Y is not written
//   EPI_AMAX   store them and fold their largest magnitude into amax_bits,
//              for a quantiser pass with a dynamic tensor scale that then
//              skips its own amax pass
constexpr int EPI_BF16 = 0, EPI_QUANT = 1, EPI_AMAX = 2;

// EPI_QUANT for one row: `tile_ok` says the row's 128-row tile exists in the
// padded scale layout; rows in it past M get their (zero) scales but no codes.
NVFP4_DEV void epi_quant_row(const W4A4Params& p, const uint32_t (&packed)[64], int row, int col0, bool tile_ok) {
  if (!tile_ok || col0 >= p.N) return;
  const float st = *p.q_st;
  const float d = __fmul_rn(st, 6.0f);
  const int nblk = min(8, (p.N - col0) / 16);   // 4 or 8 (N % 64 == 0)
  uint32_t scw[2] = {0u, 0u};
  uint4 cw[4];
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    float v[16];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t w = packed[8 * b + e];
      v[2 * e] = __uint_as_float(w << 16);
      v[2 * e + 1] = __uint_as_float(w & 0xFFFF0000u);
    }
    uint2 c;
    const uint32_t sc = quant_block16(v, st, d, c);
    scw[b >> 2] |= sc << (8 * (b & 3));
    if (b & 1) {
      cw[b >> 1].z = c.x;
      cw[b >> 1].w = c.y;
    } else {
      cw[b >> 1].x = c.x;
      cw[b >> 1].y = c.y;
    }
  }
  if (row < p.M) {
    uint4* dst = reinterpret_cast<uint4*>(p.q_codes + static_cast<int64_t>(row) * (p.N / 2) + col0 / 2);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (2 * q < nblk) dst[q] = cw[q];
  }
  // scale byte (row, c) of the MMA layout with N/16 columns (a multiple of 4):
  // ((row / 128) * (N / 64) + c / 4) * 512 + (row % 32) * 16 + ((row / 32) % 4) * 4 + c % 4
  const int c0 = col0 / 16;
#pragma unroll
  for (int g = 0; g < 2; ++g)
    if (4 * g < nblk) {
      const int c = c0 + 4 * g;
      const int64_t off = (static_cast<int64_t>(row >> 7) * (p.N / 64) + (c >> 2)) * 512 + (row & 31) * 16 +
                          ((row >> 5) & 3) * 4;
      *reinterpret_cast<uint32_t*>(p.q_scales + off) = scw[g];
    }
}

// EPI_AMAX: the warp's largest output magnitude into amax_bits.
NVFP4_DEV void epi_amax(const W4A4Params& p, const uint32_t (&packed)[64], bool valid) {
  uint32_t m = 0u;
  if (valid) {
#pragma unroll
    for (int i = 0; i < 64; ++i) m = max(m, max(packed[i] & 0x7FFFu, (packed[i] >> 16) & 0x7FFFu));
  }
  m = __reduce_max_sync(0xffffffffu, m);
  // bf16 magnitude bits order like the values; as fp32 bits they are m << 16
  if ((threadIdx.x & 31) == 0 && m != 0u) atomicMax(p.amax_bits, m << 16);
}

// tile index -> (m_tile, n_tile): bands of BAND m-tiles sweep all n-tiles,
// m fastest, so the CTAs working at one time share A and W tiles in L2
NVFP4_DEV void tile_coords(int tile, const W4A4Params& p, int& m_tile, int& n_tile) {
  const int band = tile / (BAND * p.n_tiles);
  const int band_m0 = band * BAND;
  const int band_h = min(BAND, p.m_tiles - band_m0);
  const int within = tile - band * BAND * p.n_tiles;
  m_tile = band_m0 + within % band_h;
  n_tile = within / band_h;
}

// Persistent: CTA c computes tiles c, c + gridDim.x, ...
//   warps 0, 2  TMA producers over the whole tile sequence (one continuous
//               ring; warp 0 fills the even stages, warp 2 the odd ones: one
//               issuing thread cannot keep an SM's TMA ingress busy)
//   warp 1      TMEM allocation; lane 0 issues the MMAs
//   warps 3..10 epilogue: drain the 128 x 256 fp32 accumulator (warp w reads
//               lane quarter w % 4, column half (w - 3) / 4) into packed bf16
//               registers, release the accumulator, then store
//   warps 11..14 scale warps: copy each stage's scale atoms from shared
//               memory into that stage's tensor-memory scale columns
// A warp may touch only the tensor-memory lane quarter warp % 4; every branch
// that ends in a .sync.aligned tcgen05 instruction is taken warp-uniformly.
template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_w4a4_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                     const W4A4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bar_base = base + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + STAGES * STAGE_BYTES);
  // bars: [0, S) full, [S, 2S) empty, [2S, 3S) scales in tensor memory,
  // 3S accumulator full, 3S+1 accumulator empty
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * STAGES + 3);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto sf_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + s); };
  const uint32_t accf_bar = bar_base + 8u * (3 * STAGES);
  const uint32_t acce_bar = bar_base + 8u * (3 * STAGES + 1);
  auto stage_a = [&](int s) { return base + s * STAGE_BYTES; };
  auto stage_b = [&](int s) { return base + s * STAGE_BYTES + A_BYTES; };
  auto stage_sfa = [&](int s) { return base + s * STAGE_BYTES + A_BYTES + B_BYTES; };
  auto stage_sfb = [&](int s) { return base + s * STAGE_BYTES + A_BYTES + B_BYTES + SFA_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles_total = p.m_tiles * p.n_tiles;
  const int n_k = (p.K + BK - 1) / BK;
  const int k_atoms_total = p.K / 64;
  const int64_t sf_row_stride = static_cast<int64_t>(k_atoms_total) * 512;   // bytes per 128-row scale strip

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sf_bar(s), SF_WARPS);
    }
    mbar_init(accf_bar, 1);
    mbar_init(acce_bar, EPI_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_a) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_b) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  int next_it = 0;             // producer: one past the last stage index this thread issued
  int mma_tiles = 0;           // MMA: tiles whose accumulation was issued
  const int prod = warp == 0 ? 0 : (warp == 2 ? 1 : -1);

  if (prod >= 0) {
    if (lane == 0) {
      int it = 0;
      for (int tile = blockIdx.x; tile < n_tiles_total && !*abort_flag; tile += gridDim.x) {
        int m_tile, n_tile;
        tile_coords(tile, p, m_tile, n_tile);
        bool ok = true;
        for (int ks = 0; ks < n_k; ++ks, ++it) {
          if ((it & 1) != prod) continue;
          const int s = it % STAGES;
          if (it >= STAGES &&
              !mbar_wait_bounded(empty_bar(s), ((it / STAGES) - 1) & 1, abort_flag, &g_device_status)) {
            ok = false;
            break;
          }
          const int atoms = min(4, k_atoms_total - 4 * ks);
          const uint32_t sf_bytes = static_cast<uint32_t>(atoms) * 512u;
          mbar_arrive_expect_tx(full_bar(s), A_BYTES + B_BYTES + 3u * sf_bytes);
          tma_load_2d(stage_a(s), &map_a, ks * 128, m_tile * BM, full_bar(s));
          tma_load_2d(stage_b(s), &map_b, ks * 128, n_tile * BN, full_bar(s));
          bulk_load(stage_sfa(s), p.sfa + m_tile * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes,
                    full_bar(s));
          bulk_load(stage_sfb(s), p.sfb + (2 * n_tile) * sf_row_stride + static_cast<int64_t>(ks) * 2048,
                    sf_bytes, full_bar(s));
          // the second 128-row half of a ragged last W tile has no scale atoms of its
          // own (the scale buffer is padded to 128 rows): reuse the first half's,
          // those output columns are never stored
          const int rt_hi = min(2 * n_tile + 1, (p.N + 127) / 128 - 1);
          bulk_load(stage_sfb(s) + 2048, p.sfb + rt_hi * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes,
                    full_bar(s));
          next_it = it + 1;
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0;
      for (int tile = blockIdx.x; tile < n_tiles_total && !*abort_flag; tile += gridDim.x) {
        // the epilogue must have drained the previous tile's accumulator
        if (mma_tiles > 0 && !mbar_wait_bounded(acce_bar, (mma_tiles - 1) & 1, abort_flag, &g_device_status)) break;
        tc_fence_after();
        bool ok = true;
        for (int ks = 0; ks < n_k; ++ks, ++it) {
          const int s = it % STAGES;
          // the scale warps arrive only after the stage's copies landed
          if (!mbar_wait_bounded(sf_bar(s), (it / STAGES) & 1, abort_flag, &g_device_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int atoms = min(4, k_atoms_total - 4 * ks);
          const uint32_t sf_col = tmem + SF_TMEM_BASE + s * SF_COLS_PER_STAGE;
          // descriptors by offset (the address field counts 16 bytes); a full
          // stage as straight-line code: the MMA thread's issue time per MMA
          // in a runtime-count loop exceeded what an N = 256 MMA takes
          const uint64_t adesc = smem_desc(stage_a(s), 16, 1024, 2), bdesc = smem_desc(stage_b(s), 16, 1024, 2);
          if (atoms == 4) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_mxf4nvf4(tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, sf_col + 4 * k, sf_col + 16 + 8 * k,
                              (ks > 0 || k > 0) ? 1u : 0u);
          } else {
            for (int k = 0; k < atoms; ++k)
              tc_mma_mxf4nvf4(tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, sf_col + 4 * k, sf_col + 16 + 8 * k,
                              (ks > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(empty_bar(s));
        }
        if (!ok) break;
        tc_commit(accf_bar);
        ++mma_tiles;
      }
    }
  } else if (warp < SF_WARP0) {
    const int quarter = warp & 3;
    const int half = (warp - EPI_WARP0) >> 2;
    const float scale = p.st_a[0] * p.st_b[0];
    int done = 0;
    for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x, ++done) {
      int m_tile, n_tile;
      tile_coords(tile, p, m_tile, n_tile);
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(accf_bar, done & 1, abort_flag, &g_device_status))) break;
      tc_fence_after();
      uint32_t packed[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc_ld_32cols(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(half * 128 + 32 * c), r);
        tc_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q)
          packed[16 * c + q] = f32x2_to_bf16x2(__uint_as_float(r[2 * q]) * scale, __uint_as_float(r[2 * q + 1]) * scale);
      }
      // the accumulator is free for the next tile's MMAs
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar);
      const int row = m_tile * BM + quarter * 32 + lane;
      const int col0 = n_tile * BN + half * 128;
      if (EPI == EPI_QUANT) {
        epi_quant_row(p, packed, row, col0, true);
        continue;
      }
      if (EPI == EPI_AMAX) epi_amax(p, packed, row < p.M && col0 < p.N);
      if (row < p.M && col0 < p.N) {
        uint16_t* dst = p.Y + static_cast<int64_t>(row) * p.N + col0;
        const int nq = (p.N - col0) >= 128 ? 16 : (p.N - col0) / 8;   // 16-byte pieces in range
#pragma unroll
        for (int q = 0; q < 16; ++q)
          if (q < nq)
            reinterpret_cast<uint4*>(dst)[q] =
                make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      }
    }
  } else {
    // Scale warps. Stage layout of the scale columns: [4k, 4k + 4) atom k of
    // A, [16 + 8k, 16 + 8k + 8) atom k of W's two 128-row halves. Lane l of
    // every lane quarter holds line l of each atom, whose four 32-bit words are
    // the four K-scales of rows l, l + 32, l + 64, l + 96 (the MMA reads the
    // word of its own quarter).
    const uint32_t lane_cols = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + SF_TMEM_BASE;
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      bool ok = true;
      for (int ks = 0; ks < n_k; ++ks, ++it) {
        const int s = it % STAGES;
        if (!__all_sync(0xffffffffu,
                        mbar_wait_bounded(full_bar(s), (it / STAGES) & 1, abort_flag, &g_device_status))) {
          ok = false;
          break;
        }
        uint32_t v[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 x = lds128(stage_sfa(s) + 512 * k + 16 * lane);
          v[4 * k] = x.x, v[4 * k + 1] = x.y, v[4 * k + 2] = x.z, v[4 * k + 3] = x.w;
        }
        const uint32_t col = lane_cols + s * SF_COLS_PER_STAGE;
        tc_st_16cols(col, v);
#pragma unroll
        for (int pair = 0; pair < 2; ++pair) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 x = lds128(stage_sfb(s) + 2048 * h + 512 * (2 * pair + kk) + 16 * lane);
              const int o = 8 * kk + 4 * h;
              v[o] = x.x, v[o + 1] = x.y, v[o + 2] = x.z, v[o + 3] = x.w;
            }
          tc_st_16cols(col + 16 + 16 * pair, v);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sf_bar(s));
      }
      if (!ok) break;
    }
  }

  // Unwind. After a give-up, let the copies and MMAs already issued land
  // (bounded) before the shared and tensor memory they target go away.
  if (prod >= 0 && lane == 0 && *abort_flag) {
    // the stages of this producer that may still be in flight: its last ones
    for (int it = next_it - 1; it >= 0 && it >= next_it - 2 * STAGES; --it)
      if ((it & 1) == prod)
        mbar_wait_bounded(full_bar(it % STAGES), (it / STAGES) & 1, nullptr, &g_device_status, 100000000ull);
  }
  if (warp == 1 && lane == 0 && *abort_flag && mma_tiles > 0) {
    mbar_wait_bounded(accf_bar, (mma_tiles - 1) & 1, nullptr, &g_device_status, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------------------
// CTA-pair version (cta_group::2), used once M spans two 128-row tiles.
//
// Each SM receives TMA data at about 55 bytes per clock whatever the other
// SMs do (measured on GB300 with L2-resident tiles), so with one CTA per
// 128 x 256 tile the 54 KB a stage brings in takes longer than the four MMAs
// it feeds. Two CTAs of a cluster share one 256 x 256 tile: each holds its
// own 128 rows of A and one 128-row half of the W tile, and one thread of the
// even CTA issues tcgen05.mma.cta_group::2 (M = 256), which reads both CTAs'
// shared memory and accumulates each CTA's 128 rows into that CTA's tensor
// memory. Per stage an SM now takes in 38 KB (A 16, W half 16, the A scales
// 2 and the whole W tile's scales 4) for the same MMA work.
//
// Synchronisation, per CTA unless stated:
//   full[s]   TMA bytes of this CTA's stage s landed (its producers)
//   ready[s]  in the even CTA only: both CTAs' scale warps have put stage s's
//             scales into their tensor memory (8 arrivals, 4 remote)
//   empty[s]  the pair's MMAs have consumed stage s (one multicast commit)
//   accf      the tile's accumulation is complete (one multicast commit)
//   acce      in the even CTA only: both CTAs' epilogues have drained the
//             accumulator (16 arrivals, 8 remote)
// Every wait is bounded; both CTAs reach the closing cluster barrier on every
// path, so a CTA never leaves while its peer may still touch its memory.
//
// The epilogue stores through TMA: each epilogue warp writes its 32 rows x 64
// columns of bf16 into a 4 KB staging box in shared memory and one lane
// issues a tensor store. A lane's plain 16-byte stores would each touch a
// different row (32 cache lines per warp instruction), and that stream of
// scattered stores held up the other warps' shared-memory traffic (measured:
// the epilogue cost a third of the run time).
constexpr int P_STAGES = 5;
constexpr int P_B_BYTES = 128 * 128;                                   // one 128-row half of the W tile
constexpr int P_STAGE_BYTES = A_BYTES + P_B_BYTES + SFA_BYTES + SFB_BYTES;   // 38 KB
// output staging: per epilogue warp 32 rows x 64 bf16 (one 128B-swizzled TMA store box)
constexpr int P_OUT_BYTES = 32 * 128;
constexpr int P_SMEM_BYTES = P_STAGES * P_STAGE_BYTES + EPI_WARPS * P_OUT_BYTES + 1024 + 256;
static_assert(SF_TMEM_BASE + P_STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "tensor memory columns");
static_assert((3 * P_STAGES + 4) * 8 <= 256, "barrier area");
constexpr int P_BAND = 16;                                             // m-pairs that share one sweep over W
// kind::mxf4nvf4, E2M1 x E2M1, K-major, N = 256, M = 256 (the pair)
constexpr uint32_t P_IDESC = (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(256 >> 4) << 24);

// Bounded wait on a barrier that threads of the peer CTA arrive on.
NVFP4_DEV bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait_cluster_bounded(bar, parity, abort_flag, &g_device_status);
}

NVFP4_DEV void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t sfa, uint32_t sfb,
                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %6, [%3], [%4], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(sfa), "r"(sfb), "r"(accumulate), "r"(P_IDESC)
      : "memory");
}

// pair tile -> (m_pair, n_tile): bands of P_BAND m-pairs sweep all n-tiles
NVFP4_DEV void pair_coords(int tile, int m_pairs, int n_tiles, int& m_pair, int& n_tile) {
  const int band = tile / (P_BAND * n_tiles);
  const int band_m0 = band * P_BAND;
  const int band_h = min(P_BAND, m_pairs - band_m0);
  const int within = tile - band * P_BAND * n_tiles;
  m_pair = band_m0 + within % band_h;
  n_tile = within / band_h;
}

// Warp roles as in gemm_w4a4_kernel, in both CTAs; in the odd CTA warp 1 only
// takes part in the tensor-memory allocation.
template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_w4a4_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                          const __grid_constant__ CUtensorMap map_y, const W4A4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t out_base = base + P_STAGES * P_STAGE_BYTES;   // 1024-aligned staging boxes
  const uint32_t bar_base = out_base + EPI_WARPS * P_OUT_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + P_STAGES * P_STAGE_BYTES + EPI_WARPS * P_OUT_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * P_STAGES + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * P_STAGES + 3);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (P_STAGES + s); };
  auto ready_bar = [&](int s) { return bar_base + 8u * (2 * P_STAGES + s); };
  const uint32_t accf_bar = bar_base + 8u * (3 * P_STAGES);
  const uint32_t acce_bar = bar_base + 8u * (3 * P_STAGES + 1);
  auto stage_a = [&](int s) { return base + s * P_STAGE_BYTES; };
  auto stage_b = [&](int s) { return base + s * P_STAGE_BYTES + A_BYTES; };
  auto stage_sfa = [&](int s) { return base + s * P_STAGE_BYTES + A_BYTES + P_B_BYTES; };
  auto stage_sfb = [&](int s) { return base + s * P_STAGE_BYTES + A_BYTES + P_B_BYTES + SFA_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair_id = static_cast<int>(blockIdx.x >> 1), n_pairs = static_cast<int>(gridDim.x >> 1);
  const int m_pairs = (p.m_tiles + 1) / 2;
  const int n_tiles_total = m_pairs * p.n_tiles;
  const int n_k = (p.K + BK - 1) / BK;
  const int k_atoms_total = p.K / 64;
  const int64_t sf_row_stride = static_cast<int64_t>(k_atoms_total) * 512;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(ready_bar(s), 2 * SF_WARPS);
    }
    mbar_init(accf_bar, 1);
    mbar_init(acce_bar, 2 * EPI_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_a) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_b) : "memory");
    if (EPI != EPI_QUANT) asm volatile("prefetch.tensormap [%0];" ::"l"(&map_y) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();   // both CTAs' barriers and tensor memory exist before anything refers to them
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  int next_it = 0;
  int mma_tiles = 0;
  const int prod = warp == 0 ? 0 : (warp == 2 ? 1 : -1);

  if (prod >= 0) {
    if (lane == 0) {
      int it = 0;
      for (int tile = pair_id; tile < n_tiles_total && !*abort_flag; tile += n_pairs) {
        int m_pair, n_tile;
        pair_coords(tile, m_pairs, p.n_tiles, m_pair, n_tile);
        const int m_tile = 2 * m_pair + static_cast<int>(rank);
        // an odd CTA past the last m-tile reads the last real scale strip; its rows are never stored
        const int rt_a = min(m_tile, p.m_tiles - 1);
        const int rt_b0 = 2 * n_tile;
        const int rt_b1 = min(2 * n_tile + 1, (p.N + 127) / 128 - 1);
        bool ok = true;
        for (int ks = 0; ks < n_k; ++ks, ++it) {
          if ((it & 1) != prod) continue;
          const int s = it % P_STAGES;
          if (it >= P_STAGES && !mbar_wait_cluster(empty_bar(s), ((it / P_STAGES) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const int atoms = min(4, k_atoms_total - 4 * ks);
          const uint32_t sf_bytes = static_cast<uint32_t>(atoms) * 512u;
          mbar_arrive_expect_tx(full_bar(s), A_BYTES + P_B_BYTES + 3u * sf_bytes);
          tma_load_2d(stage_a(s), &map_a, ks * 128, m_tile * BM, full_bar(s));
          tma_load_2d(stage_b(s), &map_b, ks * 128, n_tile * BN + static_cast<int>(rank) * 128, full_bar(s));
          bulk_load(stage_sfa(s), p.sfa + rt_a * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes,
                    full_bar(s));
          bulk_load(stage_sfb(s), p.sfb + rt_b0 * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes,
                    full_bar(s));
          bulk_load(stage_sfb(s) + 2048, p.sfb + rt_b1 * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes,
                    full_bar(s));
          next_it = it + 1;
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      int it = 0;
      for (int tile = pair_id; tile < n_tiles_total && !*abort_flag; tile += n_pairs) {
        // both CTAs' epilogues must have drained the previous tile's accumulator
        if (mma_tiles > 0 && !mbar_wait_cluster(acce_bar, (mma_tiles - 1) & 1, abort_flag)) break;
        tc_fence_after();
        bool ok = true;
        for (int ks = 0; ks < n_k; ++ks, ++it) {
          const int s = it % P_STAGES;
          // both CTAs' scale warps arrive only after their stage's copies landed
          if (!mbar_wait_cluster(ready_bar(s), (it / P_STAGES) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int atoms = min(4, k_atoms_total - 4 * ks);
          const uint32_t sf_col = tmem + SF_TMEM_BASE + s * SF_COLS_PER_STAGE;
          // descriptors by offset (the address field counts 16 bytes); a full
          // stage as straight-line code (see gemm_w4a4_kernel). This costs the
          // bf16-output instantiation a 40-byte spill (register cap 128 at
          // 512 threads), measured cheaper than the runtime-count loop.
          const uint64_t adesc = smem_desc(stage_a(s), 16, 1024, 2), bdesc = smem_desc(stage_b(s), 16, 1024, 2);
          if (atoms == 4) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_pair(tmem, adesc + 2 * k, bdesc + 2 * k, sf_col + 4 * k, sf_col + 16 + 8 * k,
                          (ks > 0 || k > 0) ? 1u : 0u);
          } else {
            for (int k = 0; k < atoms; ++k)
              tc_mma_pair(tmem, adesc + 2 * k, bdesc + 2 * k, sf_col + 4 * k, sf_col + 16 + 8 * k,
                          (ks > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit_pair(empty_bar(s));
        }
        if (!ok) break;
        tc_commit_pair(accf_bar);
        ++mma_tiles;
      }
    }
  } else if (warp < SF_WARP0) {
    const int quarter = warp & 3;
    const int half = (warp - EPI_WARP0) >> 2;
    const float scale = p.st_a[0] * p.st_b[0];
    int done = 0;
    for (int tile = pair_id; tile < n_tiles_total; tile += n_pairs, ++done) {
      int m_pair, n_tile;
      pair_coords(tile, m_pairs, p.n_tiles, m_pair, n_tile);
      if (!__all_sync(0xffffffffu, mbar_wait_cluster(accf_bar, done & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t packed[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc_ld_32cols(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(half * 128 + 32 * c), r);
        tc_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q)
          packed[16 * c + q] = f32x2_to_bf16x2(__uint_as_float(r[2 * q]) * scale, __uint_as_float(r[2 * q + 1]) * scale);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_bar, 0);
      const int row0 = (2 * m_pair + static_cast<int>(rank)) * BM + quarter * 32;
      const int col0 = n_tile * BN + half * 128;
      if (EPI == EPI_QUANT) {
        epi_quant_row(p, packed, row0 + lane, col0, 2 * m_pair + static_cast<int>(rank) < p.m_tiles);
        continue;
      }
      if (EPI == EPI_AMAX) epi_amax(p, packed, 2 * m_pair + static_cast<int>(rank) < p.m_tiles && row0 + lane < p.M);
      // two 64-column boxes through this warp's staging buffer (128B swizzle:
      // 16-byte chunk c of row r at r * 128 + (c ^ (r % 8)) * 16)
      const uint32_t stage_out = out_base + static_cast<uint32_t>(warp - EPI_WARP0) * P_OUT_BYTES;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        // the previous box's store has finished reading the staging buffer
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t a = stage_out + lane * 128 + ((c ^ (lane & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(packed[32 * b + 4 * c]),
                       "r"(packed[32 * b + 4 * c + 1]), "r"(packed[32 * b + 4 * c + 2]), "r"(packed[32 * b + 4 * c + 3])
                       : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the tensor store
        __syncwarp();
        if (lane == 0 && row0 < p.M && col0 + 64 * b < p.N) {
          asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(&map_y),
                       "r"(col0 + 64 * b), "r"(row0), "r"(stage_out)
                       : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      }
    }
    // stores complete before the CTA exits
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  } else {
    // scale warps: this CTA's A scales and the whole W tile's scales into its
    // own tensor memory (layout as in gemm_w4a4_kernel), then tell the even CTA
    const uint32_t lane_cols = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + SF_TMEM_BASE;
    int it = 0;
    for (int tile = pair_id; tile < n_tiles_total; tile += n_pairs) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      bool ok = true;
      for (int ks = 0; ks < n_k; ++ks, ++it) {
        const int s = it % P_STAGES;
        if (!__all_sync(0xffffffffu,
                        mbar_wait_bounded(full_bar(s), (it / P_STAGES) & 1, abort_flag, &g_device_status))) {
          ok = false;
          break;
        }
        uint32_t v[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 x = lds128(stage_sfa(s) + 512 * k + 16 * lane);
          v[4 * k] = x.x, v[4 * k + 1] = x.y, v[4 * k + 2] = x.z, v[4 * k + 3] = x.w;
        }
        const uint32_t col = lane_cols + s * SF_COLS_PER_STAGE;
        tc_st_16cols(col, v);
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 x = lds128(stage_sfb(s) + 2048 * h + 512 * (2 * pr + kk) + 16 * lane);
              const int o = 8 * kk + 4 * h;
              v[o] = x.x, v[o + 1] = x.y, v[o + 2] = x.z, v[o + 3] = x.w;
            }
          tc_st_16cols(col + 16 + 16 * pr, v);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(ready_bar(s), 0);
      }
      if (!ok) break;
    }
  }

  // Unwind: copies and MMAs already issued land (bounded) before the memory they target goes away.
  if (prod >= 0 && lane == 0 && *abort_flag) {
    for (int it = next_it - 1; it >= 0 && it >= next_it - 2 * P_STAGES; --it)
      if ((it & 1) == prod)
        mbar_wait_bounded(full_bar(it % P_STAGES), (it / P_STAGES) & 1, nullptr, &g_device_status, 100000000ull);
  }
  if (warp == 1 && rank == 0 && lane == 0 && *abort_flag && mma_tiles > 0) {
    mbar_wait_bounded(accf_bar, (mma_tiles - 1) & 1, nullptr, &g_device_status, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // the peer is done with this CTA's shared and tensor memory
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// One CTA waits on an mbarrier that nothing arrives on: the bounded wait must
// give up, record NVFP4_ERR_TIMEOUT and free the tensor memory it took.
__global__ void bounded_wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t slot;
  __shared__ int abort_flag;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&slot)), "r"(32)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) mbar_wait_bounded(b, 0, &abort_flag, &g_device_status, limit_ns);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(slot), "r"(32) : "memory");
}

// ---------------------------------------------------------------------------
// Routed experts with 4-bit activations (W4A4 MoE): a persistent grouped GEMM
// over the routing plan's tile table, on the same block-scaled FP4 mainloop
// and warp roles as gemm_w4a4_kernel. The routed rows' NVFP4 codes sit in a
// tile-major matrix (tile t = up to 128 routed rows of one expert at rows
// [128 t, 128 t + 128), the rest of the tile zero), so each tile is one TMA
// box and one strip of the MMA scale layout. Work item w = (tile w / n_tiles,
// weight block w % n_tiles); the tile count is read on the device.
//   GATEUP  W13 [E][2I][H]: weight block j = gate rows [128 j, 128 j + 128)
//           and the matching up rows I + [128 j, ...) in one 256-column
//           accumulator; epilogue h = bf16(silu(g) * u) into the routed rows'
//           h buffer (padded row order of the plan) and the largest |h| into
//           amax_bits (the dynamic tensor scale of the h rows)
//   DOWN    W2 [E][H][I]: weight block j = rows [256 j, 256 j + 256);
//           epilogue y (bf16) per routed row for the combine
struct GroupedW4A4Params {
  const uint8_t* sfa;             // MMA-layout scales of the tile-major routed rows
  const uint8_t* sfb;             // MMA-layout scales of each expert matrix, expert e at e * sfb_expert_bytes
  int64_t sfb_expert_bytes;
  const float* st_a;              // [1] the routed rows' tensor scale
  const float* st_b;              // [E] the experts' tensor scales
  const int* tile_count;
  const int* tile_expert;
  const int* tile_row0;           // first row of the tile in the plan's padded row order
  const int* tile_rows;
  int K;                          // H (gate/up) or I (down)
  int n_tiles;                    // weight blocks per tile: I / 128 (gate/up) or H / 256 (down)
  int rows_per_expert;            // 2I or H
  int inter;                      // I
  int hidden;                     // H
  uint16_t* h_out;                // GATEUP: bf16 [padded rows][I]
  unsigned int* amax_bits;        // GATEUP: max |h| as fp32 bits (zero on entry)
  uint16_t* y_out;                // DOWN: bf16 [padded rows][H]
};

template <bool GATEUP>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_w4a4_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const GroupedW4A4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bar_base = base + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * STAGES + 3);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto sf_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + s); };
  const uint32_t accf_bar = bar_base + 8u * (3 * STAGES);
  const uint32_t acce_bar = bar_base + 8u * (3 * STAGES + 1);
  auto stage_a = [&](int s) { return base + s * STAGE_BYTES; };
  auto stage_b = [&](int s) { return base + s * STAGE_BYTES + A_BYTES; };
  auto stage_sfa = [&](int s) { return base + s * STAGE_BYTES + A_BYTES + B_BYTES; };
  auto stage_sfb = [&](int s) { return base + s * STAGE_BYTES + A_BYTES + B_BYTES + SFA_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_work = *p.tile_count * p.n_tiles;
  const int n_k = (p.K + BK - 1) / BK;
  const int k_atoms_total = p.K / 64;
  const int64_t sf_row_stride = static_cast<int64_t>(k_atoms_total) * 512;   // bytes per 128-row scale strip

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sf_bar(s), SF_WARPS);
    }
    mbar_init(accf_bar, 1);
    mbar_init(acce_bar, EPI_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_a) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_b) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  int next_it = 0;
  int mma_tiles = 0;
  const int prod = warp == 0 ? 0 : (warp == 2 ? 1 : -1);

  if (prod >= 0) {
    if (lane == 0) {
      int it = 0;
      for (int w = blockIdx.x; w < n_work && !*abort_flag; w += gridDim.x) {
        const int t = w / p.n_tiles, j = w - t * p.n_tiles;
        const int e = p.tile_expert[t];
        // the two 128-row weight boxes and their scale strips within expert e
        const int rb0 = GATEUP ? j : 2 * j;
        const int rb1 = GATEUP ? p.inter / 128 + j : 2 * j + 1;
        const int ybase = e * p.rows_per_expert;
        const uint8_t* sfb_e = p.sfb + static_cast<int64_t>(e) * p.sfb_expert_bytes;
        bool ok = true;
        for (int ks = 0; ks < n_k; ++ks, ++it) {
          if ((it & 1) != prod) continue;
          const int s = it % STAGES;
          if (it >= STAGES &&
              !mbar_wait_bounded(empty_bar(s), ((it / STAGES) - 1) & 1, abort_flag, &g_device_status)) {
            ok = false;
            break;
          }
          const int atoms = min(4, k_atoms_total - 4 * ks);
          const uint32_t sf_bytes = static_cast<uint32_t>(atoms) * 512u;
          mbar_arrive_expect_tx(full_bar(s), A_BYTES + B_BYTES + 3u * sf_bytes);
          tma_load_2d(stage_a(s), &map_a, ks * 128, t * BM, full_bar(s));
          // expert weights, streamed about once per call: evicted from L2
          // first, so h and the per-slot outputs stay there for the kernels
          // that read them next (T=256: 0.113 -> 0.104 ms per layer; with
          // 256-row tiles on CTA pairs, where those outputs outgrow L2, the
          // same policy measured slower and is not used)
          const uint64_t pol = l2_policy_evict_first();
          tma_load_2d_hint(stage_b(s), &map_b, ks * 128, ybase + rb0 * 128, full_bar(s), pol);
          tma_load_2d_hint(stage_b(s) + B_BYTES / 2, &map_b, ks * 128, ybase + rb1 * 128, full_bar(s), pol);
          bulk_load(stage_sfa(s), p.sfa + t * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes, full_bar(s));
          bulk_load(stage_sfb(s), sfb_e + rb0 * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes,
                    full_bar(s));
          bulk_load(stage_sfb(s) + 2048, sfb_e + rb1 * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes,
                    full_bar(s));
          next_it = it + 1;
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0;
      for (int w = blockIdx.x; w < n_work && !*abort_flag; w += gridDim.x) {
        if (mma_tiles > 0 && !mbar_wait_bounded(acce_bar, (mma_tiles - 1) & 1, abort_flag, &g_device_status)) break;
        tc_fence_after();
        bool ok = true;
        for (int ks = 0; ks < n_k; ++ks, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait_bounded(sf_bar(s), (it / STAGES) & 1, abort_flag, &g_device_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int atoms = min(4, k_atoms_total - 4 * ks);
          const uint32_t sf_col = tmem + SF_TMEM_BASE + s * SF_COLS_PER_STAGE;
          // descriptors by offset (the address field counts 16 bytes); a full
          // stage as straight-line code: the MMA thread's issue time per MMA
          // in a runtime-count loop exceeded what an N = 256 MMA takes
          const uint64_t adesc = smem_desc(stage_a(s), 16, 1024, 2), bdesc = smem_desc(stage_b(s), 16, 1024, 2);
          if (atoms == 4) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_mxf4nvf4(tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, sf_col + 4 * k, sf_col + 16 + 8 * k,
                              (ks > 0 || k > 0) ? 1u : 0u);
          } else {
            for (int k = 0; k < atoms; ++k)
              tc_mma_mxf4nvf4(tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, sf_col + 4 * k, sf_col + 16 + 8 * k,
                              (ks > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(empty_bar(s));
        }
        if (!ok) break;
        tc_commit(accf_bar);
        ++mma_tiles;
      }
    }
  } else if (warp < SF_WARP0) {
    const int quarter = warp & 3;
    const int half = (warp - EPI_WARP0) >> 2;
    const int i = quarter * 32 + lane;                 // row within the tile
    int done = 0;
    for (int w = blockIdx.x; w < n_work; w += gridDim.x, ++done) {
      const int t = w / p.n_tiles, j = w - t * p.n_tiles;
      const int e = p.tile_expert[t];
      const int nrows = p.tile_rows[t];
      const int64_t row = static_cast<int64_t>(p.tile_row0[t]) + i;
      const float scale = p.st_a[0] * p.st_b[e];
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(accf_bar, done & 1, abort_flag, &g_device_status))) break;
      tc_fence_after();
      const uint32_t lanes = static_cast<uint32_t>(quarter * 32) << 16;
      if (GATEUP) {
        // intermediate columns [64 half, 64 half + 64) of block j: gate at
        // accumulator columns 64 half + c, up at 128 + 64 half + c
        uint32_t hv[32];
        uint32_t hmax = 0u;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t g[32], u[32];
          tc_ld_32cols(tmem + lanes + static_cast<uint32_t>(64 * half + 32 * c), g);
          tc_ld_32cols(tmem + lanes + static_cast<uint32_t>(128 + 64 * half + 32 * c), u);
          tc_wait_ld();
          if (c == 1) {
            // the accumulator's last reads: the next item's MMAs may start
            // while this warp does the SiLU math and the stores
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar);
          }
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float g0 = __uint_as_float(g[2 * q]) * scale, g1 = __uint_as_float(g[2 * q + 1]) * scale;
            const float u0 = __uint_as_float(u[2 * q]) * scale, u1 = __uint_as_float(u[2 * q + 1]) * scale;
            // silu with the fast exponential and division (relative error ~1e-7,
            // far below the bf16 rounding of h); this math sits between the MMAs
            // of one work item and the next, since the accumulator is not double
            // buffered (tensor memory is full)
            const uint32_t b = f32x2_to_bf16x2(__fdividef(g0, 1.0f + __expf(-g0)) * u0,
                                               __fdividef(g1, 1.0f + __expf(-g1)) * u1);
            hv[16 * c + q] = b;
            hmax = max(hmax, max(b & 0x7FFFu, (b >> 16) & 0x7FFFu));
          }
        }
        const bool valid = i < nrows;
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.h_out + row * p.inter + j * 128 + 64 * half);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_uint4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
        }
        const uint32_t m = __reduce_max_sync(0xffffffffu, valid ? hmax : 0u);
        if (lane == 0 && m != 0u) atomicMax(p.amax_bits, m << 16);
      } else {
        // the row's 128 columns are read and packed to bf16 before any store,
        // and the accumulator released then: with the stores between the
        // reads the next item's MMAs waited for them (70% of the MMA thread's
        // time in the down GEMM)
        uint4* dst = reinterpret_cast<uint4*>(p.y_out + row * p.hidden + j * 256 + half * 128);
        uint32_t packed[64];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tc_ld_32cols(tmem + lanes + static_cast<uint32_t>(half * 128 + 32 * c), r);
          tc_wait_ld();
#pragma unroll
          for (int q = 0; q < 16; ++q)
            packed[16 * c + q] = f32x2_to_bf16x2(__uint_as_float(r[2 * q]) * scale, __uint_as_float(r[2 * q + 1]) * scale);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar);
        if (i < nrows) {
#pragma unroll
          for (int q = 0; q < 16; ++q)
            dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
        }
      }
    }
  } else {
    // scale warps, as in gemm_w4a4_kernel
    const uint32_t lane_cols = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + SF_TMEM_BASE;
    int it = 0;
    for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      bool ok = true;
      for (int ks = 0; ks < n_k; ++ks, ++it) {
        const int s = it % STAGES;
        if (!__all_sync(0xffffffffu,
                        mbar_wait_bounded(full_bar(s), (it / STAGES) & 1, abort_flag, &g_device_status))) {
          ok = false;
          break;
        }
        uint32_t v[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 x = lds128(stage_sfa(s) + 512 * k + 16 * lane);
          v[4 * k] = x.x, v[4 * k + 1] = x.y, v[4 * k + 2] = x.z, v[4 * k + 3] = x.w;
        }
        const uint32_t col = lane_cols + s * SF_COLS_PER_STAGE;
        tc_st_16cols(col, v);
#pragma unroll
        for (int pair = 0; pair < 2; ++pair) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 x = lds128(stage_sfb(s) + 2048 * h + 512 * (2 * pair + kk) + 16 * lane);
              const int o = 8 * kk + 4 * h;
              v[o] = x.x, v[o + 1] = x.y, v[o + 2] = x.z, v[o + 3] = x.w;
            }
          tc_st_16cols(col + 16 + 16 * pair, v);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sf_bar(s));
      }
      if (!ok) break;
    }
  }

  // Unwind after a give-up: copies and MMAs already issued land (bounded)
  // before the shared and tensor memory they target go away.
  if (prod >= 0 && lane == 0 && *abort_flag) {
    for (int it = next_it - 1; it >= 0 && it >= next_it - 2 * STAGES; --it)
      if ((it & 1) == prod)
        mbar_wait_bounded(full_bar(it % STAGES), (it / STAGES) & 1, nullptr, &g_device_status, 100000000ull);
  }
  if (warp == 1 && lane == 0 && *abort_flag && mma_tiles > 0) {
    mbar_wait_bounded(accf_bar, (mma_tiles - 1) & 1, nullptr, &g_device_status, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// Issue-rate ceiling of the block-scaled FP4 tensor cores: one CTA per SM
// issues `n_mma` tcgen05.mma.kind::mxf4nvf4 of 128 x 256 x 64 (the W4A4
// kernels' instruction) back to back into one accumulator, operands from
// shared memory (zeros) and block scales from tensor memory, no global
// memory traffic; the tensor pipe is the only thing it can wait on. Timed by
// the caller, it gives the FP4 rate this part reaches, for the W4A4 GEMM's
// roofline beside the nominal figure. The completion wait is bounded.
constexpr int PROBE_THREADS = 128;
// more shared memory than two CTAs could share, so each SM holds one CTA and
// no CTA waits for another's tensor memory
constexpr int PROBE_SMEM = 120 * 1024;
static_assert(A_BYTES + B_BYTES + 1024 + 64 <= PROBE_SMEM && 2 * PROBE_SMEM > 228 * 1024, "probe shared memory");
__global__ void __launch_bounds__(PROBE_THREADS, 1) fp4_mma_rate_kernel(int n_mma) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bar = base + A_BYTES + B_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + A_BYTES + B_BYTES + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + A_BYTES + B_BYTES + 16);
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (A_BYTES + B_BYTES) / 16; i += PROBE_THREADS)
    reinterpret_cast<uint4*>(base_ptr)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the zeros are visible to the tensor pipe
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  {
    // zero scale columns (E4M3 0 is a finite scale): each warp its lane quarter
    uint32_t z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0u;
    const uint32_t lane_cols = tmem + (static_cast<uint32_t>(warp * 32) << 16) + SF_TMEM_BASE;
    tc_st_16cols(lane_cols, z);
    tc_st_16cols(lane_cols + 16, z);
    tc_st_16cols(lane_cols + 32, z);
    tc_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint64_t adesc = smem_desc(base, 16, 1024, 2);
    const uint64_t bdesc = smem_desc(base + A_BYTES, 16, 1024, 2);
    for (int i = 0; i < n_mma; ++i)
      tc_mma_mxf4nvf4(tmem, adesc, bdesc, IDESC, tmem + SF_TMEM_BASE, tmem + SF_TMEM_BASE + 16, i > 0 ? 1u : 0u);
    tc_commit(bar);
    mbar_wait_bounded(bar, 0, abort_flag, &g_device_status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// 2-D map over packed codes [rows][K/2] bytes, 128 x 128-byte boxes, 128B swizzle.
int make_code_map(CUtensorMap* map, const uint8_t* codes, int64_t rows, int64_t K, int box_rows) {
  return make_tmap_2d_u8(map, codes, K / 2, rows, K / 2, 128, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

}  // namespace

size_t w4a4_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return align_up(static_cast<size_t>(mma_scale_rows(M) * mma_scale_cols(K))) +
         align_up(static_cast<size_t>(mma_scale_rows(N) * mma_scale_cols(K)));
}

namespace {

template <int EPI>
int launch_w4a4_epi(const nvfp4_tensor_t& A, const nvfp4_tensor_t& W, uint16_t* Y, void* ws, cudaStream_t stream,
                    uint8_t* q_codes, uint8_t* q_scales, const float* q_st, unsigned int* amax_bits) {
  const int64_t M = A.rows, N = W.rows, K = A.K;
  if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  const uint8_t* sfa = A.scales;
  const uint8_t* sfb = W.scales;
  char* w = static_cast<char*>(ws);
  if (A.scale_layout == NVFP4_SCALES_ROWMAJOR) {
    uint8_t* dst = reinterpret_cast<uint8_t*>(w);
    int rc = launch_prepack_scales(A.scales, 1, M, K, dst, stream);
    if (rc != NVFP4_OK) return rc;
    sfa = dst;
  }
  if (W.scale_layout == NVFP4_SCALES_ROWMAJOR) {
    uint8_t* dst =
        reinterpret_cast<uint8_t*>(w + align_up(static_cast<size_t>(mma_scale_rows(M) * mma_scale_cols(K))));
    int rc = launch_prepack_scales(W.scales, 1, N, K, dst, stream);
    if (rc != NVFP4_OK) return rc;
    sfb = dst;
  }
  CUtensorMap map_a, map_b;
  int rc = make_code_map(&map_a, A.codes, M, K, BM);
  if (rc != NVFP4_OK) return rc;
  rc = make_code_map(&map_b, W.codes, N, K, BN);
  if (rc != NVFP4_OK) return rc;

  rc = ensure_smem(gemm_w4a4_kernel<EPI>, SMEM_BYTES);
  if (rc != NVFP4_OK) return rc;
  W4A4Params p{};
  p.q_codes = q_codes;
  p.q_scales = q_scales;
  p.q_st = q_st;
  p.amax_bits = amax_bits;
  p.sfa = sfa;
  p.sfb = sfb;
  p.st_a = A.s_t;
  p.st_b = W.s_t;
  p.Y = Y;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.m_tiles = static_cast<int>(ceil_div(M, BM));
  p.n_tiles = static_cast<int>(ceil_div(N, BN));
  if (p.m_tiles >= 2) {
    // CTA pairs on 256 x 256 tiles: W tiles come in 128-row halves
    rc = make_code_map(&map_b, W.codes, N, K, 128);
    if (rc != NVFP4_OK) return rc;
    rc = ensure_smem(gemm_w4a4_pair_kernel<EPI>, P_SMEM_BYTES);
    if (rc != NVFP4_OK) return rc;
    // bf16 Y [M][N]: stores of 64 columns x 32 rows (N % 8 == 0 keeps the row stride 16-byte aligned);
    // the quantising epilogue writes no Y and never touches the map
    CUtensorMap map_y{};
    if (EPI != EPI_QUANT) {
      rc = make_tmap_2d_u16(&map_y, Y, N, M, N * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc != NVFP4_OK) return rc;
    }
    const int64_t pair_tiles = ceil_div(p.m_tiles, 2) * p.n_tiles;
    const int64_t max_pairs = sm_count() / 2;
    const unsigned grid = static_cast<unsigned>(2 * (pair_tiles < max_pairs ? pair_tiles : max_pairs));
    return launch_ex(gemm_w4a4_pair_kernel<EPI>, dim3(grid), dim3(THREADS), P_SMEM_BYTES, 2, false, stream, map_a,
                     map_b, map_y, p);
  }
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
  const unsigned grid = static_cast<unsigned>(tiles < sm_count() ? tiles : sm_count());
  gemm_w4a4_kernel<EPI><<<grid, THREADS, SMEM_BYTES, stream>>>(map_a, map_b, p);
  return from_cuda(cudaGetLastError());
}

// The grouped expert GEMM on CTA pairs (cta_group::2), as gemm_w4a4_pair_kernel
// does for one matrix: a work item is (tile t of up to 256 routed rows of one
// expert, weight block j of 256 rows); the even CTA takes routed rows
// [0, 128) of the tile and the odd one [128, 256), each loads one 128-row half
// of the weight block (gate/up: the gate rows in the even CTA, the matching
// up rows in the odd one; down: rows [256 j, +128) and [256 j + 128, +128)),
// both hold the whole block's scales, and the even CTA's thread issues the
// M = 256 MMAs. Per stage an SM now takes in 38 KB where the one-CTA kernel
// took 54 KB for the same MMA work (the copies bound it). The routed rows are
// tile-major with 256-row tiles (128-row MMA-layout scale strips 2t, 2t + 1).
// Epilogue per warp (32 routed rows, one lane quarter): read and pack the
// accumulator, release it, then store through a 4 KB staging box and a TMA
// store (128B swizzle), or with plain stores where the box would reach past
// the tile's rows (the next tile's rows follow in the plan's order).
template <bool GATEUP>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_w4a4_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                             const __grid_constant__ CUtensorMap map_out, const GroupedW4A4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t out_base = base + P_STAGES * P_STAGE_BYTES;   // 1024-aligned staging boxes
  const uint32_t bar_base = out_base + EPI_WARPS * P_OUT_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + P_STAGES * P_STAGE_BYTES + EPI_WARPS * P_OUT_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * P_STAGES + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * P_STAGES + 3);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (P_STAGES + s); };
  auto ready_bar = [&](int s) { return bar_base + 8u * (2 * P_STAGES + s); };
  const uint32_t accf_bar = bar_base + 8u * (3 * P_STAGES);
  const uint32_t acce_bar = bar_base + 8u * (3 * P_STAGES + 1);
  auto stage_a = [&](int s) { return base + s * P_STAGE_BYTES; };
  auto stage_b = [&](int s) { return base + s * P_STAGE_BYTES + A_BYTES; };
  auto stage_sfa = [&](int s) { return base + s * P_STAGE_BYTES + A_BYTES + P_B_BYTES; };
  auto stage_sfb = [&](int s) { return base + s * P_STAGE_BYTES + A_BYTES + P_B_BYTES + SFA_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair_id = static_cast<int>(blockIdx.x >> 1), n_pairs = static_cast<int>(gridDim.x >> 1);
  const int n_work = *p.tile_count * p.n_tiles;
  const int n_k = (p.K + BK - 1) / BK;
  const int k_atoms_total = p.K / 64;
  const int64_t sf_row_stride = static_cast<int64_t>(k_atoms_total) * 512;   // bytes per 128-row scale strip

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(ready_bar(s), 2 * SF_WARPS);
    }
    mbar_init(accf_bar, 1);
    mbar_init(acce_bar, 2 * EPI_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_a) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_b) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_out) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();   // both CTAs' barriers and tensor memory exist before anything refers to them
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  int next_it = 0;
  int mma_tiles = 0;
  const int prod = warp == 0 ? 0 : (warp == 2 ? 1 : -1);

  if (prod >= 0) {
    if (lane == 0) {
      int it = 0;
      for (int w = pair_id; w < n_work && !*abort_flag; w += n_pairs) {
        const int t = w / p.n_tiles, j = w - t * p.n_tiles;
        const int e = p.tile_expert[t];
        const int strip = 2 * t + static_cast<int>(rank);   // this CTA's 128 routed rows
        // the weight block's two 128-row halves and their scale strips within expert e
        const int rb0 = GATEUP ? j : 2 * j;
        const int rb1 = GATEUP ? p.inter / 128 + j : 2 * j + 1;
        const int ybase = e * p.rows_per_expert;
        const int my_rb = rank == 0 ? rb0 : rb1;
        const uint8_t* sfb_e = p.sfb + static_cast<int64_t>(e) * p.sfb_expert_bytes;
        bool ok = true;
        for (int ks = 0; ks < n_k; ++ks, ++it) {
          if ((it & 1) != prod) continue;
          const int s = it % P_STAGES;
          if (it >= P_STAGES && !mbar_wait_cluster(empty_bar(s), ((it / P_STAGES) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const int atoms = min(4, k_atoms_total - 4 * ks);
          const uint32_t sf_bytes = static_cast<uint32_t>(atoms) * 512u;
          mbar_arrive_expect_tx(full_bar(s), A_BYTES + P_B_BYTES + 3u * sf_bytes);
          tma_load_2d(stage_a(s), &map_a, ks * 128, strip * BM, full_bar(s));
          tma_load_2d(stage_b(s), &map_b, ks * 128, ybase + my_rb * 128, full_bar(s));
          bulk_load(stage_sfa(s), p.sfa + strip * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes,
                    full_bar(s));
          bulk_load(stage_sfb(s), sfb_e + rb0 * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes,
                    full_bar(s));
          bulk_load(stage_sfb(s) + 2048, sfb_e + rb1 * sf_row_stride + static_cast<int64_t>(ks) * 2048, sf_bytes,
                    full_bar(s));
          next_it = it + 1;
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      int it = 0;
      for (int w = pair_id; w < n_work && !*abort_flag; w += n_pairs) {
        // both CTAs' epilogues must have read the previous item's accumulator
        if (mma_tiles > 0 && !mbar_wait_cluster(acce_bar, (mma_tiles - 1) & 1, abort_flag)) break;
        tc_fence_after();
        bool ok = true;
        for (int ks = 0; ks < n_k; ++ks, ++it) {
          const int s = it % P_STAGES;
          // both CTAs' scale warps arrive only after their stage's copies landed
          if (!mbar_wait_cluster(ready_bar(s), (it / P_STAGES) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int atoms = min(4, k_atoms_total - 4 * ks);
          const uint32_t sf_col = tmem + SF_TMEM_BASE + s * SF_COLS_PER_STAGE;
          const uint64_t adesc = smem_desc(stage_a(s), 16, 1024, 2), bdesc = smem_desc(stage_b(s), 16, 1024, 2);
          if (atoms == 4) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_pair(tmem, adesc + 2 * k, bdesc + 2 * k, sf_col + 4 * k, sf_col + 16 + 8 * k,
                          (ks > 0 || k > 0) ? 1u : 0u);
          } else {
            for (int k = 0; k < atoms; ++k)
              tc_mma_pair(tmem, adesc + 2 * k, bdesc + 2 * k, sf_col + 4 * k, sf_col + 16 + 8 * k,
                          (ks > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit_pair(empty_bar(s));
        }
        if (!ok) break;
        tc_commit_pair(accf_bar);
        ++mma_tiles;
      }
    }
  } else if (warp < SF_WARP0) {
    const int quarter = warp & 3;
    const int half = (warp - EPI_WARP0) >> 2;
    const uint32_t lanes = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t stage_out = out_base + static_cast<uint32_t>(warp - EPI_WARP0) * P_OUT_BYTES;
    int done = 0;
    for (int w = pair_id; w < n_work; w += n_pairs, ++done) {
      const int t = w / p.n_tiles, j = w - t * p.n_tiles;
      const int e = p.tile_expert[t];
      const int nrows = p.tile_rows[t];
      const int li0 = 128 * static_cast<int>(rank) + 32 * quarter;   // this warp's first row within the tile
      const int li = li0 + lane;
      const bool valid = li < nrows;
      const int64_t row0 = static_cast<int64_t>(p.tile_row0[t]) + li0;   // plan row of lane 0
      const float scale = p.st_a[0] * p.st_b[e];
      if (!__all_sync(0xffffffffu, mbar_wait_cluster(accf_bar, done & 1, abort_flag))) break;
      tc_fence_after();
      // packed bf16 outputs of this lane's row: gate/up 64 h values (columns
      // 128 j + 64 half ..), down 128 y values (columns 256 j + 128 half ..)
      constexpr int NW = GATEUP ? 32 : 64;
      uint32_t packed[NW];
      uint32_t hmax = 0u;
      if (GATEUP) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t g[32], u[32];
          tc_ld_32cols(tmem + lanes + static_cast<uint32_t>(64 * half + 32 * c), g);
          tc_ld_32cols(tmem + lanes + static_cast<uint32_t>(128 + 64 * half + 32 * c), u);
          tc_wait_ld();
          if (c == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce_bar, 0);
          }
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float g0 = __uint_as_float(g[2 * q]) * scale, g1 = __uint_as_float(g[2 * q + 1]) * scale;
            const float u0 = __uint_as_float(u[2 * q]) * scale, u1 = __uint_as_float(u[2 * q + 1]) * scale;
            const uint32_t b = f32x2_to_bf16x2(__fdividef(g0, 1.0f + __expf(-g0)) * u0,
                                               __fdividef(g1, 1.0f + __expf(-g1)) * u1);
            packed[16 * c + q] = b;
            hmax = max(hmax, max(b & 0x7FFFu, (b >> 16) & 0x7FFFu));
          }
        }
        const uint32_t m = __reduce_max_sync(0xffffffffu, valid ? hmax : 0u);
        if (lane == 0 && m != 0u) atomicMax(p.amax_bits, m << 16);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tc_ld_32cols(tmem + lanes + static_cast<uint32_t>(half * 128 + 32 * c), r);
          tc_wait_ld();
#pragma unroll
          for (int q = 0; q < 16; ++q)
            packed[16 * c + q] = f32x2_to_bf16x2(__uint_as_float(r[2 * q]) * scale, __uint_as_float(r[2 * q + 1]) * scale);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acce_bar, 0);
      }
      const int col0 = GATEUP ? 128 * j + 64 * half : 256 * j + 128 * half;
      if (li0 + 32 <= nrows) {
        // 64-column boxes through this warp's staging buffer (128B swizzle:
        // 16-byte chunk c of row r at r * 128 + (c ^ (r % 8)) * 16)
#pragma unroll
        for (int b = 0; b < NW / 32; ++b) {
          // the previous box's store has finished reading the staging buffer
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t a = stage_out + lane * 128 + ((c ^ (lane & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(packed[32 * b + 4 * c]),
                         "r"(packed[32 * b + 4 * c + 1]), "r"(packed[32 * b + 4 * c + 2]),
                         "r"(packed[32 * b + 4 * c + 3])
                         : "memory");
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the tensor store
          __syncwarp();
          if (lane == 0) {
            asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(&map_out),
                         "r"(col0 + 64 * b), "r"(static_cast<int>(row0)), "r"(stage_out)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        }
      } else if (valid) {
        // the tile's ragged last rows: plain stores of this lane's row
        uint4* dst = reinterpret_cast<uint4*>((GATEUP ? p.h_out + (row0 + lane) * p.inter
                                                      : p.y_out + (row0 + lane) * p.hidden) + col0);
#pragma unroll
        for (int q = 0; q < NW / 4; ++q)
          dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      }
    }
    // stores complete before the CTA exits
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  } else {
    // scale warps: this CTA's A scales and the whole weight block's scales
    // into its own tensor memory (layout as in gemm_w4a4_kernel), then tell
    // the even CTA
    const uint32_t lane_cols = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + SF_TMEM_BASE;
    int it = 0;
    for (int w = pair_id; w < n_work; w += n_pairs) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      bool ok = true;
      for (int ks = 0; ks < n_k; ++ks, ++it) {
        const int s = it % P_STAGES;
        if (!__all_sync(0xffffffffu,
                        mbar_wait_bounded(full_bar(s), (it / P_STAGES) & 1, abort_flag, &g_device_status))) {
          ok = false;
          break;
        }
        uint32_t v[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 x = lds128(stage_sfa(s) + 512 * k + 16 * lane);
          v[4 * k] = x.x, v[4 * k + 1] = x.y, v[4 * k + 2] = x.z, v[4 * k + 3] = x.w;
        }
        const uint32_t col = lane_cols + s * SF_COLS_PER_STAGE;
        tc_st_16cols(col, v);
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 x = lds128(stage_sfb(s) + 2048 * h + 512 * (2 * pr + kk) + 16 * lane);
              const int o = 8 * kk + 4 * h;
              v[o] = x.x, v[o + 1] = x.y, v[o + 2] = x.z, v[o + 3] = x.w;
            }
          tc_st_16cols(col + 16 + 16 * pr, v);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(ready_bar(s), 0);
      }
      if (!ok) break;
    }
  }

  // Unwind: copies and MMAs already issued land (bounded) before the memory they target goes away.
  if (prod >= 0 && lane == 0 && *abort_flag) {
    for (int it = next_it - 1; it >= 0 && it >= next_it - 2 * P_STAGES; --it)
      if ((it & 1) == prod)
        mbar_wait_bounded(full_bar(it % P_STAGES), (it / P_STAGES) & 1, nullptr, &g_device_status, 100000000ull);
  }
  if (warp == 1 && rank == 0 && lane == 0 && *abort_flag && mma_tiles > 0) {
    mbar_wait_bounded(accf_bar, (mma_tiles - 1) & 1, nullptr, &g_device_status, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // the peer is done with this CTA's shared and tensor memory
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

}  // namespace

int launch_gemm_w4a4(const nvfp4_tensor_t& A, const nvfp4_tensor_t& W, uint16_t* Y, void* ws,
                     cudaStream_t stream) {
  return launch_w4a4_epi<EPI_BF16>(A, W, Y, ws, stream, nullptr, nullptr, nullptr, nullptr);
}

size_t w4a4_quant_workspace_bytes(int64_t M, int64_t N, int64_t K) { return w4a4_workspace_bytes(M, N, K) + 256; }

// W4A4 whose output is handed on as NVFP4 (MMA-layout scales). GIVEN: one
// fused kernel. COMPUTE: the GEMM writes the bf16 output and its amax, then
// the quantiser encodes it with s_t = amax / 2688, skipping its own amax pass.
int launch_gemm_w4a4_quant(const nvfp4_tensor_t& A, const nvfp4_tensor_t& W, uint8_t* codes, uint8_t* scales,
                           float* s_t, int s_t_mode, uint16_t* Y, void* ws, cudaStream_t stream) {
  unsigned int* amax = reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + w4a4_workspace_bytes(A.rows, W.rows, A.K));
  if (s_t_mode == NVFP4_ST_GIVEN)
    return launch_w4a4_epi<EPI_QUANT>(A, W, nullptr, ws, stream, codes, scales, s_t, nullptr);
  if (cudaMemsetAsync(amax, 0, sizeof(unsigned int), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  int rc = launch_w4a4_epi<EPI_AMAX>(A, W, Y, ws, stream, nullptr, nullptr, nullptr, amax);
  if (rc != NVFP4_OK) return rc;
  return launch_quantize_bf16_from_amax(Y, A.rows, W.rows, codes, scales, amax, s_t, stream);
}

int read_device_status(int* out, cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
  *out = v;
  return NVFP4_OK;
}

int launch_grouped_w4a4(bool gateup, const uint8_t* a_codes, const uint8_t* a_scales, const float* st_a,
                        int64_t a_rows, const nvfp4_tensor_t& W, const int* tile_count, const int* tile_expert,
                        const int* tile_row0, const int* tile_rows, int64_t max_tiles, int inter, int hidden,
                        uint16_t* h_out, unsigned int* amax_bits, uint16_t* y_out, int64_t out_rows, bool pair,
                        cudaStream_t stream) {
  const int64_t K = W.K, rows = static_cast<int64_t>(W.batch) * W.rows;
  CUtensorMap map_a, map_b, map_out;
  int rc = make_tmap_2d_u8(&map_a, a_codes, K / 2, a_rows, K / 2, 128, BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != NVFP4_OK) return rc;
  rc = make_tmap_2d_u8(&map_b, W.codes, K / 2, rows, K / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != NVFP4_OK) return rc;
  // the output rows in the plan's order, 32-row x 64-column boxes
  rc = gateup ? make_tmap_2d_u16(&map_out, h_out, inter, out_rows, static_cast<int64_t>(inter) * 2, 64, 32,
                                 CU_TENSOR_MAP_SWIZZLE_128B)
              : make_tmap_2d_u16(&map_out, y_out, hidden, out_rows, static_cast<int64_t>(hidden) * 2, 64, 32,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != NVFP4_OK) return rc;
  GroupedW4A4Params p{};
  p.sfa = a_scales;
  p.sfb = W.scales;
  p.sfb_expert_bytes = mma_scale_rows(W.rows) * mma_scale_cols(K);
  p.st_a = st_a;
  p.st_b = W.s_t;
  p.tile_count = tile_count;
  p.tile_expert = tile_expert;
  p.tile_row0 = tile_row0;
  p.tile_rows = tile_rows;
  p.K = static_cast<int>(K);
  p.n_tiles = gateup ? inter / 128 : hidden / 256;
  p.rows_per_expert = static_cast<int>(W.rows);
  p.inter = inter;
  p.hidden = hidden;
  p.h_out = h_out;
  p.amax_bits = amax_bits;
  p.y_out = y_out;
  const int64_t work_max = max_tiles * p.n_tiles;
  if (!pair) {
    // persistent: at most one CTA per SM, fewer when the plan cannot have that many work items
    const unsigned grid = static_cast<unsigned>(work_max < sm_count() ? work_max : sm_count());
    if (gateup) {
      rc = ensure_smem(grouped_w4a4_kernel<true>, SMEM_BYTES);
      if (rc != NVFP4_OK) return rc;
      grouped_w4a4_kernel<true><<<grid, THREADS, SMEM_BYTES, stream>>>(map_a, map_b, p);
    } else {
      rc = ensure_smem(grouped_w4a4_kernel<false>, SMEM_BYTES);
      if (rc != NVFP4_OK) return rc;
      grouped_w4a4_kernel<false><<<grid, THREADS, SMEM_BYTES, stream>>>(map_a, map_b, p);
    }
    return from_cuda(cudaGetLastError());
  }
  // persistent CTA pairs: at most one CTA per SM, fewer when the plan cannot have that many work items
  const int64_t pairs_max = sm_count() / 2;
  const unsigned grid = static_cast<unsigned>(2 * (work_max < pairs_max ? work_max : pairs_max));
  if (gateup) {
    rc = ensure_smem(grouped_w4a4_pair_kernel<true>, P_SMEM_BYTES);
    if (rc != NVFP4_OK) return rc;
    return launch_ex(grouped_w4a4_pair_kernel<true>, dim3(grid), dim3(THREADS), P_SMEM_BYTES, 2, false, stream,
                     map_a, map_b, map_out, p);
  }
  rc = ensure_smem(grouped_w4a4_pair_kernel<false>, P_SMEM_BYTES);
  if (rc != NVFP4_OK) return rc;
  return launch_ex(grouped_w4a4_pair_kernel<false>, dim3(grid), dim3(THREADS), P_SMEM_BYTES, 2, false, stream,
                   map_a, map_b, map_out, p);
}

int probe_fp4_mma_rate(int n_mma, int n_ctas, cudaStream_t stream) {
  int rc = ensure_smem(fp4_mma_rate_kernel, PROBE_SMEM);
  if (rc != NVFP4_OK) return rc;
  const int grid = n_ctas > 0 ? n_ctas : sm_count();
  fp4_mma_rate_kernel<<<grid, PROBE_THREADS, PROBE_SMEM, stream>>>(n_mma);
  return from_cuda(cudaGetLastError());
}

int selftest_bounded_wait(int64_t limit_ns, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<unsigned long long>(limit_ns));
  return from_cuda(cudaGetLastError());
}

}  // namespace nvfp4
