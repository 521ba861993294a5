// Skinny W4A16 mainloop shared by the decode GEMV, the masked draft head and
// the routed-expert MoE layer.
//
// Shape of the work. Weights W[rows][K] are NVFP4 (codes [rows][K/2], E4M3
// scales [rows][K/16], row-major); activations are up to 32 rows ("tokens")
// of 16-bit values. Each CTA owns 128 weight rows (8 warps x 16) and one
// chunk of 32 tokens, over a range of K; a warp streams its 16 rows with
// 128-bit loads, 128 K-elements (64 bytes per row) per iteration, dequantises
// in registers (cvt e2m1x2 -> f16x2, times the E4M3 scale in f16, which is
// exact: |code * scale| <= 2688 with at most six significant bits) and feeds
// mma.sync m16n8k16 with fp32 accumulation: the weight rows are the MMA's M
// side, tokens its N side.
//
// K order inside an iteration is permuted so that each lane's 16 loaded bytes
// are exactly its MMA A-fragments: lane (g, t) loads bytes [16t, 16t+16) of
// rows g and g+8, i.e. K elements [32t, 32t+32), and uses bytes (2j, 2j+1) in
// MMA j; the activations are stored in the matching order by the prep kernel,
// so the permutation cancels in the dot product.
//
// Activations reach the tensor cores as f16: the prep kernel multiplies each
// token by 2^-p (p from the token's amax, putting it in [2^14, 2^15)), which
// is exact for every element above amax * 2^-29 and keeps the f16 range; the
// epilogue multiplies by 2^p again.
#pragma once

#include "common.cuh"

namespace nvfp4 {

constexpr int GV_THREADS = 256;   // 8 warps
constexpr int GV_ROWS = 128;      // weight rows per CTA
constexpr int GV_KIT = 128;       // K elements per iteration
constexpr int GV_MCHUNK = 32;     // tokens per chunk (4 n-tiles of 8)
constexpr int GV_PF = 3;          // iterations of weights in flight per warp
constexpr int GV_NTS = 4;         // n-tile slots per chunk in the fragment layout

// Fragment-major activation layout, 16-byte units:
//   [chunk][it][nt (4)][w (4)][lane (32)]
// unit (c, it, nt, w, g*4+t) holds f16 elements k = it*128 + 32t + 8w + (0..7)
// of token c*32 + nt*8 + g.
NVFP4_DEV int64_t xfrag_unit(int64_t chunk, int64_t n_it, int64_t it, int nt, int w, int lane) {
  return (((chunk * n_it + it) * GV_NTS + nt) * 4 + w) * 32 + lane;
}
inline size_t xfrag_bytes(int64_t chunks, int64_t K) {
  return static_cast<size_t>(chunks) * static_cast<size_t>(K / GV_KIT) * GV_NTS * 4 * 32 * 16;
}

// Convert one activation row into the fragment layout.
//   src     bf16 row of K elements, or nullptr for a padding row (zeros)
//   out_row index of the row in chunk order (chunk = out_row / 32)
// Writes p (the power-of-two shift) to pexp[out_row]. One CTA per row.
NVFP4_DEV void xprep_row(const uint16_t* src, int64_t K, int64_t out_row, uint4* xfrag, int* pexp) {
  __shared__ float red[32];
  const int tid = threadIdx.x;
  const int64_t n8 = K / 8;
  float amax = 0.f;
  if (src != nullptr) {
    for (int64_t q = tid; q < n8; q += blockDim.x) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + q);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w4[e] & 0xFFFFu)));
        amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w4[e] >> 16)));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  if (tid < 32) {
    float v = tid < static_cast<int>(blockDim.x / 32) ? red[tid] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (tid == 0) red[0] = v;
  }
  __syncthreads();
  amax = red[0];
  int p = 0;
  if (amax > 0.f) p = min(max(ilogbf(amax) - 14, -100), 113);
  const float mul = ldexpf(1.0f, -p);
  if (tid == 0) pexp[out_row] = p;

  const int64_t chunk = out_row / GV_MCHUNK;
  const int nt = static_cast<int>((out_row % GV_MCHUNK) / 8);
  const int g = static_cast<int>(out_row % 8);
  const int64_t n_it = K / GV_KIT;
  for (int64_t q = tid; q < n8; q += blockDim.x) {
    uint4 o = make_uint4(0, 0, 0, 0);
    if (src != nullptr) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + q);
      o.x = f32x2_to_f16x2(bf16_bits_to_f32(v.x & 0xFFFFu) * mul, bf16_bits_to_f32(v.x >> 16) * mul);
      o.y = f32x2_to_f16x2(bf16_bits_to_f32(v.y & 0xFFFFu) * mul, bf16_bits_to_f32(v.y >> 16) * mul);
      o.z = f32x2_to_f16x2(bf16_bits_to_f32(v.z & 0xFFFFu) * mul, bf16_bits_to_f32(v.z >> 16) * mul);
      o.w = f32x2_to_f16x2(bf16_bits_to_f32(v.w & 0xFFFFu) * mul, bf16_bits_to_f32(v.w >> 16) * mul);
    }
    const int64_t it = q / 16;
    const int rem = static_cast<int>(q % 16);
    const int t = rem / 4, w = rem % 4;
    xfrag[xfrag_unit(chunk, n_it, it, nt, w, g * 4 + t)] = o;
  }
}

// Single-pass version of xprep_row for K <= 8 * 4 * blockDim.x: every thread
// keeps its (up to four) 16-byte chunks in registers between the amax and the
// conversion, so the row is read from memory once.
template <int CHUNKS>
NVFP4_DEV void xprep_row_regs(const uint16_t* src, int64_t K, int64_t out_row, uint4* xfrag, int* pexp) {
  __shared__ float red[32];
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int64_t n8 = K / 8;
  uint4 v[CHUNKS];
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    const int64_t q = tid + static_cast<int64_t>(c) * nthr;
    v[c] = make_uint4(0, 0, 0, 0);
    if (src != nullptr && q < n8) v[c] = __ldg(reinterpret_cast<const uint4*>(src) + q);
    const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w4[e] & 0xFFFFu)));
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w4[e] >> 16)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  if (tid < 32) {
    float r = tid < nthr / 32 ? red[tid] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, o));
    if (tid == 0) red[0] = r;
  }
  __syncthreads();
  amax = red[0];
  int p = 0;
  if (amax > 0.f) p = min(max(ilogbf(amax) - 14, -100), 113);
  const float mul = ldexpf(1.0f, -p);
  if (tid == 0) pexp[out_row] = p;
  const int64_t chunk = out_row / GV_MCHUNK;
  const int nt = static_cast<int>((out_row % GV_MCHUNK) / 8);
  const int g = static_cast<int>(out_row % 8);
  const int64_t n_it = K / GV_KIT;
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    const int64_t q = tid + static_cast<int64_t>(c) * nthr;
    if (q < n8) {
      uint4 o;
      o.x = f32x2_to_f16x2(bf16_bits_to_f32(v[c].x & 0xFFFFu) * mul, bf16_bits_to_f32(v[c].x >> 16) * mul);
      o.y = f32x2_to_f16x2(bf16_bits_to_f32(v[c].y & 0xFFFFu) * mul, bf16_bits_to_f32(v[c].y >> 16) * mul);
      o.z = f32x2_to_f16x2(bf16_bits_to_f32(v[c].z & 0xFFFFu) * mul, bf16_bits_to_f32(v[c].z >> 16) * mul);
      o.w = f32x2_to_f16x2(bf16_bits_to_f32(v[c].w & 0xFFFFu) * mul, bf16_bits_to_f32(v[c].w >> 16) * mul);
      const int64_t it = q / 16;
      const int rem = static_cast<int>(q % 16);
      xfrag[xfrag_unit(chunk, n_it, it, nt, rem % 4, g * 4 + rem / 4)] = o;
    }
  }
}

// The mainloop: accumulate the 16 rows of this warp (rows g and g+8 of the
// lane) against NT n-tiles of tokens over iterations [0, nit).
//   cA, cB   code bytes of rows g, g+8 at this warp's first iteration,
//            already offset by 16*t
//   sA, sB   scale bytes of rows g, g+8 at the first iteration, offset 2*t
//   xf       fragment units of (chunk, first iteration), lane offset applied
template <int NT>
NVFP4_DEV void gemv_mainloop(float (&acc)[NT][4], const uint8_t* cA, const uint8_t* cB,
                             const uint8_t* sA, const uint8_t* sB, const uint4* xf, int nit) {
  uint4 ra[GV_PF], rb[GV_PF];
  uint32_t qa[GV_PF], qb[GV_PF];
#pragma unroll
  for (int d = 0; d < GV_PF; ++d) {
    if (d < nit) {
      ra[d] = ld_stream_v4(cA + d * 64);
      rb[d] = ld_stream_v4(cB + d * 64);
      qa[d] = ld_stream_u16(sA + d * 8);
      qb[d] = ld_stream_u16(sB + d * 8);
    }
  }
  for (int i0 = 0; i0 < nit; i0 += GV_PF) {
#pragma unroll
    for (int d = 0; d < GV_PF; ++d) {
      const int i = i0 + d;
      if (i < nit) {
        const uint32_t wa[4] = {ra[d].x, ra[d].y, ra[d].z, ra[d].w};
        const uint32_t wb[4] = {rb[d].x, rb[d].y, rb[d].z, rb[d].w};
        const uint32_t scA = e4m3x2_to_f16x2(qa[d]);
        const uint32_t scB = e4m3x2_to_f16x2(qb[d]);
        if (i + GV_PF < nit) {
          ra[d] = ld_stream_v4(cA + (i + GV_PF) * 64);
          rb[d] = ld_stream_v4(cB + (i + GV_PF) * 64);
          qa[d] = ld_stream_u16(sA + (i + GV_PF) * 8);
          qb[d] = ld_stream_u16(sB + (i + GV_PF) * 8);
        }
        const uint4* xi = xf + static_cast<int64_t>(i) * (GV_NTS * 4 * 32);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t fa[4], fb[4];
          e2m1x8_to_f16x2(wa[w], fa);
          e2m1x8_to_f16x2(wb[w], fb);
          // bytes 0..7 of the lane's 16 use the first block scale, 8..15 the second
          const uint32_t sa = w < 2 ? dup_lo(scA) : dup_hi(scA);
          const uint32_t sb = w < 2 ? dup_lo(scB) : dup_hi(scB);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            fa[e] = hmul2(fa[e], sa);
            fb[e] = hmul2(fb[e], sb);
          }
          const uint32_t A0[4] = {fa[0], fb[0], fa[1], fb[1]};
          const uint32_t A1[4] = {fa[2], fb[2], fa[3], fb[3]};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint4 bx = __ldg(xi + (nt * 4 + w) * 32);
            mma_f16_16816(acc[nt], A0, bx.x, bx.y);
            mma_f16_16816(acc[nt], A1, bx.z, bx.w);
          }
        }
      }
    }
  }
}

// SK_GATEUP_DENSE: a dense gate/up projection W [2I][K] (gate rows [0, I),
// up rows [I, 2I)) whose epilogue writes h = bf16(silu(g) * u) [M][I].
enum SkinnyMode { SK_PLAIN = 0, SK_ARGMAX = 1, SK_MOE_GATEUP = 2, SK_MOE_DOWN = 3, SK_GATEUP_DENSE = 4 };

struct SkinnyParams {
  // weights (row-major scales); batched tensors use global row ids
  const uint8_t* codes;
  const uint8_t* scales;
  const float* s_t;
  int64_t K;
  int64_t n_rows;              // PLAIN: N; ARGMAX: number of candidate rows
  const int32_t* idx;          // ARGMAX: candidate -> vocabulary row (nullable)
  int64_t w_rows;              // ARGMAX: rows of the weight; an idx entry outside [0, w_rows) is skipped
  // activations in fragment layout and their per-row power-of-two shifts
  const uint4* xfrag;
  const int* pexp;
  int64_t M;                   // PLAIN / ARGMAX tokens
  int split;                   // CTAs per cluster along K
  // PLAIN
  uint16_t* Y;                 // bf16 [M][N]
  // ARGMAX
  unsigned long long* keys;    // [M], zero on entry
  unsigned int* counter;       // zero on entry
  int32_t* out_ids;
  float* out_logit;
  // MoE
  const int* chunk_count;
  const int* chunk_expert;
  const int* chunk_rows;
  int64_t inter;               // I
  int64_t hidden;              // H
  int64_t rows_per_expert;     // rows of one expert matrix
  uint16_t* h_out;             // GATEUP: bf16 [padded rows][I]
  uint16_t* y_out;             // DOWN: bf16 [padded rows][H]
};

template <int NT, int MODE>
__global__ void __launch_bounds__(GV_THREADS, 2) skinny_kernel(const SkinnyParams p) {
  __shared__ __align__(16) float part[8 * NT][GV_ROWS];
  __shared__ unsigned long long kbest[GV_MCHUNK];
  __shared__ int s_last;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int S = p.split;
  const int s = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int64_t n_it = p.K / GV_KIT;
  const int it0 = static_cast<int>(n_it * s / S);
  const int nit = static_cast<int>(n_it * (s + 1) / S) - it0;

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
  if (MODE == SK_ARGMAX && tid < GV_MCHUNK) kbest[tid] = 0ull;

  // weight rows of this lane: tile rows 16*warp + g and 16*warp + g + 8
  int64_t wrow[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = warp * 16 + g + 8 * h;
    int64_t w = 0;
    if (MODE == SK_PLAIN) {
      const int64_t n = row_tile * GV_ROWS + r;
      w = n < p.n_rows ? n : 0;
    } else if (MODE == SK_ARGMAX) {
      const int64_t j = row_tile * GV_ROWS + r;
      w = j < p.n_rows ? (p.idx ? static_cast<int64_t>(p.idx[j]) : j) : 0;
      if (w < 0 || w >= p.w_rows) w = 0;   // a skipped entry reads row 0; its key is dropped below
    } else if (MODE == SK_MOE_GATEUP) {
      const int64_t rr = r < 64 ? row_tile * 64 + r : p.inter + row_tile * 64 + (r - 64);
      w = expert * p.rows_per_expert + rr;
    } else {
      const int64_t rr = row_tile * GV_ROWS + r;
      w = expert * p.rows_per_expert + (rr < p.hidden ? rr : 0);
    }
    wrow[h] = w;
  }
  const int64_t kb = p.K / 2, ks = p.K / 16;
  const uint8_t* cA = p.codes + wrow[0] * kb + static_cast<int64_t>(it0) * 64 + t * 16;
  const uint8_t* cB = p.codes + wrow[1] * kb + static_cast<int64_t>(it0) * 64 + t * 16;
  const uint8_t* sA = p.scales + wrow[0] * ks + static_cast<int64_t>(it0) * 8 + t * 2;
  const uint8_t* sB = p.scales + wrow[1] * ks + static_cast<int64_t>(it0) * 8 + t * 2;
  const uint4* xf = p.xfrag + xfrag_unit(chunk, n_it, it0, 0, 0, lane);

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;

  gemv_mainloop<NT>(acc, cA, cB, sA, sB, xf, nit);

#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) part[nt * 8 + 2 * t + (e & 1)][warp * 16 + g + 8 * (e >> 1)] = acc[nt][e];

  if (S > 1) cluster_sync_all(); else __syncthreads();

  // Reduce the split-K partials of this CTA's slice of rows and finish.
  const int slice = (GV_ROWS + S - 1) / S;
  const int r_begin = min(GV_ROWS, s * slice);
  const int r_end = min(GV_ROWS, r_begin + slice);
  const int width = (MODE == SK_MOE_GATEUP) ? 64 : (r_end - r_begin);
  const int rb = (MODE == SK_MOE_GATEUP) ? 0 : r_begin;
  const int64_t row_base = chunk * GV_MCHUNK;
  const float st = p.s_t[expert];
  for (int e = tid; e < rows_in_chunk * width; e += GV_THREADS) {
    const int tok = e / width;
    const int r = rb + e % width;
    float v = 0.f;
    if (S > 1) {
      const uint32_t sa = smem_addr(&part[tok][r]);
      for (int q = 0; q < S; ++q) v += ld_dsmem_f32(sa, q);
    } else {
      v = part[tok][r];
    }
    const float mul = ldexpf(st, p.pexp[row_base + tok]);
    if (MODE == SK_PLAIN) {
      const int64_t n = row_tile * GV_ROWS + r;
      if (n < p.n_rows) p.Y[(row_base + tok) * p.n_rows + n] = static_cast<uint16_t>(f32_to_bf16_bits(v * mul));
    } else if (MODE == SK_ARGMAX) {
      const int64_t j = row_tile * GV_ROWS + r;
      const int64_t vj = j < p.n_rows ? (p.idx ? static_cast<int64_t>(p.idx[j]) : j) : -1;
      if (vj >= 0 && vj < p.w_rows) {
        const uint32_t vid = static_cast<uint32_t>(vj);
        const unsigned long long key =
            (static_cast<unsigned long long>(float_order_key(v * mul)) << 32) | (0xFFFFFFFFu - vid);
        atomicMax(&kbest[tok], key);
      }
    } else if (MODE == SK_MOE_GATEUP) {
      const float gg = v * mul;
      const float uu = part[tok][64 + r] * mul;
      const float hh = gg / (1.0f + expf(-gg)) * uu;
      p.h_out[(row_base + tok) * p.inter + row_tile * 64 + r] = static_cast<uint16_t>(f32_to_bf16_bits(hh));
    } else {
      const int64_t c = row_tile * GV_ROWS + r;
      if (c < p.hidden) p.y_out[(row_base + tok) * p.hidden + c] = static_cast<uint16_t>(f32_to_bf16_bits(v * mul));
    }
  }
  if (S > 1) cluster_sync_all();

  if (MODE == SK_ARGMAX) {
    __syncthreads();
    if (tid < rows_in_chunk) atomicMax(&p.keys[row_base + tid], kbest[tid]);
    fence_acq_rel_gpu();
    __syncthreads();
    if (tid == 0) {
      const unsigned int total = gridDim.x * gridDim.y * gridDim.z;
      s_last = atomicAdd(p.counter, 1u) == total - 1;
    }
    __syncthreads();
    if (s_last) {
      fence_acq_rel_gpu();
      for (int64_t m = tid; m < p.M; m += GV_THREADS) {
        const unsigned long long key = atomicExch(&p.keys[m], 0ull);
        p.out_ids[m] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
        if (p.out_logit) p.out_logit[m] = float_from_order_key(static_cast<uint32_t>(key >> 32));
      }
      if (tid == 0) atomicExch(p.counter, 0u);
    }
  }
}

}  // namespace nvfp4
