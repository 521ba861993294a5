// Routed-expert MoE layer, W4A16 (What 350+ Experiments Taught Us About
// Serving Qwen 3.6 35B-A3B, sections 1 and 7: the routed-expert layout and an
// NVFP4 mixture-of-experts kernel):
//   route:    top-k of softmax(router logits), ties to the lower expert id
//   plan:     group the T*k routed rows by expert, each expert padded to a
//             multiple of 32 rows (one token chunk of the skinny kernel), in
//             one single-CTA kernel
//   gate/up:  [g; u] = x @ W13_e^T, h = bf16(silu(g) * u)
//   down:     y = bf16(h @ W2_e^T) (fp32 accumulation)
// (both on the TMA-fed skinny kernel when K is a multiple of 256, else on the
// register-fed one; with at least XT_MIN_ROWS_PER_EXPERT routed rows per
// expert on average, on the tensor cores instead: moe_tc.cuh)
//   combine:  out[t] = bf16(sum_j w[t][j] * y[pos(t, j)]) in fp32, slots in order
// The order in which routed rows land inside an expert's group comes from
// atomics, but every row's arithmetic is independent of its position, so the
// output is deterministic.
#include "gemv_core.cuh"
#include "gemv_tma.cuh"
#include "launch.h"
#include "moe_tc.cuh"
#include "quant_core.cuh"

namespace nvfp4 {

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// One warp per token: fp32 softmax over E experts, then k rounds of "largest
// (p, -id) below the previous winner".
__global__ void route_kernel(const float* logits, int64_t T, int E, int topk, int32_t* ids, float* weights) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* l = logits + t * E;
  float mx = -INFINITY;
  for (int e = lane; e < E; e += 32) mx = fmaxf(mx, l[e]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  for (int e = lane; e < E; e += 32) sum += expf(l[e] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  unsigned long long prev = ~0ull;
  for (int j = 0; j < topk; ++j) {
    unsigned long long best = 0ull;
    for (int e = lane; e < E; e += 32) {
      const float p = expf(l[e] - mx) / sum;
      const unsigned long long key =
          (static_cast<unsigned long long>(float_order_key(p)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e));
      if (key < prev && key > best) best = key;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    prev = best;
    if (lane == 0) {
      ids[t * topk + j] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(best));
      weights[t * topk + j] = float_from_order_key(static_cast<uint32_t>(best >> 32));
    }
  }
}

// The same routing with the token's probabilities held in registers (E <=
// 32 EPL): the logits are read and each probability computed once, by the
// same expressions as route_kernel, so the ids and weights are identical.
template <int EPL>
__global__ void route_reg_kernel(const float* logits, int64_t T, int E, int topk, int32_t* ids, float* weights) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* l = logits + t * E;
  float v[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? l[e] : -INFINITY;
  }
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i) mx = fmaxf(mx, v[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i < E) sum += expf(v[i] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  unsigned long long key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    const float pr = expf(v[i] - mx) / sum;
    key[i] = e < E ? (static_cast<unsigned long long>(float_order_key(pr)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e))
                   : 0ull;
  }
  unsigned long long prev = ~0ull;
  for (int j = 0; j < topk; ++j) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (key[i] < prev && key[i] > best) best = key[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    prev = best;
    if (lane == 0) {
      ids[t * topk + j] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(best));
      weights[t * topk + j] = float_from_order_key(static_cast<uint32_t>(best >> 32));
    }
  }
}

// tile sizes of the routing plan: the W4A4 expert GEMM takes tiles of up to
// 128 routed rows (its MMAs are M = 128 over routed rows), the W4A16
// tensor-core kernel tiles of up to XT_NMAX; the tile table is sized for the
// smaller
constexpr int PLAN_TILE_MIN = 128;
// the cooperative routing plan: at most this many CTAs, each with a slice of
// at least PLAN_COOP_SLICE routed slots
constexpr int PLAN_COOP_MAX_G = 128;
constexpr int PLAN_COOP_SLICE = 512;
constexpr int PLAN_COOP_THREADS = 512;
constexpr int PLAN_COOP_MAX_E = 256;

// rows of the W4A4 layer's tile-major matrices: every tile of up to
// W4A4_TILE routed rows of one expert in its own W4A4_TILE rows
inline int64_t w4a4_tile_rows(int64_t R, int64_t E) { return (ceil_div(R, W4A4_TILE) + E) * W4A4_TILE; }

struct MoeWs {
  int* chunk_count;   // [1]
  int* poff;          // [E]
  int* chunk_expert;  // [max_chunks]
  int* chunk_rows;    // [max_chunks]
  int* tile_count;    // [1]  tensor-core tiles: up to tile_max rows of one expert, split evenly
  int* tile_expert;   // [max_tiles]
  int* tile_row0;     // [max_tiles]
  int* tile_rows;     // [max_tiles]
  int* row_of;        // [padded rows] token id or -1
  int* pos_of;        // [T*k]
  int* plan_hist;     // [PLAN_COOP_MAX_G][E]: the cooperative plan's per-CTA expert counts
  unsigned int* plan_bar;   // [1]: its grid barrier
  int* pexp1;         // [padded rows]
  int* pexp2;         // [padded rows]
  uint4* xfrag1;      // tokens, K = H
  uint16_t* hbuf;     // [padded rows][I] bf16
  uint4* xfrag2;      // h, K = I
  uint16_t* ybuf;     // [padded rows][H] bf16: each routed row's expert output
  // W4A4 layer: the routed rows as NVFP4 in tile-major order (tile t = rows
  // [W4A4_TILE t, W4A4_TILE (t + 1))), codes and MMA-layout scales, for x and h
  uint8_t* xq_codes;
  uint8_t* xq_scales;
  uint8_t* xt_codes;   // the layer input quantised once per token: [T][H/2]
  uint8_t* xt_scales;  // [T][H/16], row-major
  void* q_ws;          // the quantiser's workspace
  uint8_t* hq_codes;
  uint8_t* hq_scales;
  unsigned int* amax;  // [0] x, [1] h (fp32 bits)
  float* st;           // [0] x, [1] h: the dynamic tensor scales
  size_t bytes;
  int64_t max_chunks;
  int64_t max_tiles;
};

// W4A16 (w4a4 false): the plan, the f16 fragment copies and the h / y
// buffers. W4A4: the plan, h / y and the tile-major NVFP4 routed rows.
MoeWs carve_moe(void* base, int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk, bool w4a4 = false) {
  MoeWs w{};
  const int64_t R = T * topk;
  w.max_chunks = ceil_div(R, GV_MCHUNK) + E;
  w.max_tiles = ceil_div(R, PLAN_TILE_MIN) + E;
  const int64_t rows = w.max_chunks * GV_MCHUNK;
  char* b = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = b + off;
    off += align_up(bytes);
    return p;
  };
  w.chunk_count = reinterpret_cast<int*>(take(sizeof(int)));
  w.poff = reinterpret_cast<int*>(take(E * sizeof(int)));
  w.chunk_expert = reinterpret_cast<int*>(take(w.max_chunks * sizeof(int)));
  w.chunk_rows = reinterpret_cast<int*>(take(w.max_chunks * sizeof(int)));
  w.tile_count = reinterpret_cast<int*>(take(sizeof(int)));
  w.tile_expert = reinterpret_cast<int*>(take(w.max_tiles * sizeof(int)));
  w.tile_row0 = reinterpret_cast<int*>(take(w.max_tiles * sizeof(int)));
  w.tile_rows = reinterpret_cast<int*>(take(w.max_tiles * sizeof(int)));
  w.row_of = reinterpret_cast<int*>(take(rows * sizeof(int)));
  w.pos_of = reinterpret_cast<int*>(take(R * sizeof(int)));
  w.plan_hist = reinterpret_cast<int*>(take(static_cast<size_t>(PLAN_COOP_MAX_G) * E * sizeof(int)));
  w.plan_bar = reinterpret_cast<unsigned int*>(take(sizeof(unsigned int)));
  if (!w4a4) {
    w.pexp1 = reinterpret_cast<int*>(take(rows * sizeof(int)));
    w.pexp2 = reinterpret_cast<int*>(take(rows * sizeof(int)));
    w.xfrag1 = reinterpret_cast<uint4*>(take(xfrag_bytes(w.max_chunks, H)));
  }
  w.hbuf = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(rows) * I * sizeof(uint16_t)));
  if (!w4a4) w.xfrag2 = reinterpret_cast<uint4*>(take(xfrag_bytes(w.max_chunks, I)));
  w.ybuf = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(rows) * H * sizeof(uint16_t)));
  if (w4a4) {
    const size_t trows = static_cast<size_t>(w4a4_tile_rows(R, E));
    w.xt_codes = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(T) * H / 2));
    w.xt_scales = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(T) * H / 16));
    w.q_ws = take(quantize_workspace_bytes());
    w.xq_codes = reinterpret_cast<uint8_t*>(take(trows * H / 2));
    w.xq_scales = reinterpret_cast<uint8_t*>(take(trows * H / 16));
    w.hq_codes = reinterpret_cast<uint8_t*>(take(trows * I / 2));
    w.hq_scales = reinterpret_cast<uint8_t*>(take(trows * I / 16));
    w.amax = reinterpret_cast<unsigned int*>(take(2 * sizeof(unsigned int)));
    w.st = reinterpret_cast<float*>(take(2 * sizeof(float)));
  }
  w.bytes = off;
  return w;
}

// The routed rows of the layer input in tile-major NVFP4 (the W4A4 gate/up
// GEMM's A operand), copied from the tokens' rows quantised once: one warp
// per row r = tile t' + i of tile t (tile rows per tile: 128 or W4A4_TILE);
// rows i < tile_rows[t] get their token's
// codes (K/2 bytes) and block scales (re-laid into the MMA layout, four
// scale columns per 32-bit store), the rest of the tile zeros.
__global__ void __launch_bounds__(8 * 32) gather_routed_kernel(const uint8_t* codes_in, const uint8_t* scales_in,
                                                               int64_t K, const int* row_of, const int* tile_count,
                                                               const int* tile_row0, const int* tile_rows,
                                                               uint8_t* codes, uint8_t* scales, int tile) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int t = static_cast<int>(r / tile), i = static_cast<int>(r % tile);
  if (t >= *tile_count) return;
  int tok = -1;
  if (i < tile_rows[t]) tok = row_of[static_cast<int64_t>(tile_row0[t]) + i];
  const int64_t kb = K / 2, ng = K / 64;   // 16-byte code pieces: kb / 16; scale groups of four: ng
  const uint4* src = reinterpret_cast<const uint4*>(codes_in + static_cast<int64_t>(tok < 0 ? 0 : tok) * kb);
  uint4* dst = reinterpret_cast<uint4*>(codes + r * kb);
  for (int64_t q = lane; q < kb / 16; q += 32) dst[q] = tok >= 0 ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(scales_in + static_cast<int64_t>(tok < 0 ? 0 : tok) * (K / 16));
  const int64_t srow_off = (r >> 7) * ng * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
  for (int64_t g = lane; g < ng; g += 32)
    *reinterpret_cast<uint32_t*>(scales + srow_off + g * 512) = tok >= 0 ? __ldg(ssrc + g) : 0u;
}

// NVFP4 of the routed rows in tile-major order (the W4A4 expert GEMMs' A
// operand): one warp per row r = tile t + i of tile t (128 or W4A4_TILE rows
// per tile); rows i < tile_rows[t]
// hold routed row tile_row0[t] + i of the plan (gather: its token's row of
// src; else that row of src), the rest of the tile zero codes and scales.
// The tensor scale is s_t = amax / 2688 (1 if amax is 0), written to
// *s_t_out; each block takes the quantiser's step (quant_core.cuh).
constexpr int QR_WARPS = 8;
__global__ void __launch_bounds__(QR_WARPS * 32) quantize_routed_kernel(const uint16_t* src, int64_t K, bool gather,
                                                                         const int* row_of, const int* tile_count,
                                                                         const int* tile_row0, const int* tile_rows,
                                                                         const unsigned int* amax_bits, float* s_t_out,
                                                                         uint8_t* codes, uint8_t* scales, int tile) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * QR_WARPS + (threadIdx.x >> 5);
  const int t = static_cast<int>(r / tile), i = static_cast<int>(r % tile);
  if (t >= *tile_count) return;
  const float amax = __uint_as_float(*amax_bits);
  const float st = amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
  if (r == 0 && lane == 0) *s_t_out = st;
  const float d = __fmul_rn(st, 6.0f);
  const uint16_t* srow = nullptr;
  if (i < tile_rows[t]) {
    const int64_t pr = static_cast<int64_t>(tile_row0[t]) + i;
    if (!gather) {
      srow = src + pr * K;
    } else {
      const int tok = row_of[pr];
      if (tok >= 0) srow = src + static_cast<int64_t>(tok) * K;
    }
  }
  const int nb = static_cast<int>(K / 16);   // a multiple of 4 (K % 64 == 0): no scale-column padding
  uint2* crow = reinterpret_cast<uint2*>(codes + r * (K / 2));
  const int64_t srow_off = (r >> 7) * (nb / 4) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
  for (int b = lane; b < nb; b += 32) {
    uint2 c = make_uint2(0u, 0u);
    uint32_t sc = 0u;
    if (srow) {
      const uint4* s4 = reinterpret_cast<const uint4*>(srow + 16 * b);
      const uint4 w0 = __ldg(s4), w1 = __ldg(s4 + 1);
      const uint32_t u[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      float v[16];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[2 * e] = __uint_as_float(u[e] << 16);
        v[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
      }
      sc = quant_block16(v, st, d, c);
    }
    crow[b] = c;
    scales[srow_off + (b >> 2) * 512 + (b & 3)] = static_cast<uint8_t>(sc);
  }
}

constexpr int PLAN_MAX_E = 4096;
// average routed rows per expert from which the expert GEMMs run on the tensor
// cores (128 experts, top-8, H = 2048, I = 768: 16 rows per expert 0.158 ms
// on the skinny kernel against 0.169 on the tensor cores, 32 rows 0.226
// against 0.183)
constexpr int XT_MIN_ROWS_PER_EXPERT = 32;

// The whole routing plan in one CTA: count the routed rows per expert (shared
// atomics, four id loads in flight per thread), pad each expert to a multiple
// of 32 rows and take the exclusive prefix sums of the padded rows and of the
// tensor-core tiles (each expert's rows in tiles of up to tile_max) with a
// block scan, write the chunk and tile tables and row_of = -1, then hand out
// each routed row's position within its expert (shared atomics again).
// Replaces a memset and three kernels (count, plan, scatter). A routed slot
// whose expert id lies outside [0, E) gets no row (pos_of = -1, so it
// contributes nothing) and sets NVFP4_ERR_INVALID_ARG in the status word.
//
// With PRIVATE (E <= PLAN_PRIVATE_MAX_E) every warp counts into its own
// histogram in dynamic shared memory (many routed rows share few experts, so
// one shared counter per expert serialised the atomics of all 1024 threads);
// each warp's histogram then becomes its exclusive offset within the expert,
// and in the position pass the warp hands out positions from there. With
// SMEM_ROWS (R + 32 E <= PLAN_SMEM_ROWS_MAX) the padded rows' token ids
// (row_of) are assembled in shared memory and written out with coalesced
// stores: tens of thousands of scattered 4-byte stores from one SM took
// longer than the rest of the plan together.
constexpr int PLAN_THREADS = 1024;
constexpr int PLAN_PRIVATE_MAX_E = 256;
constexpr int PLAN_SMEM_ROWS_MAX = 40960;
template <bool PRIVATE, bool SMEM_ROWS>
__global__ void __launch_bounds__(PLAN_THREADS) route_plan_kernel(const int32_t* ids, int64_t R, int topk, int E,
                                                                  int* poff, int* chunk_count, int* chunk_expert,
                                                                  int* chunk_rows, int* tile_count, int* tile_expert,
                                                                  int* tile_row0, int* tile_rows, int* row_of,
                                                                  int* pos_of, int* status, int tile_max) {
  __shared__ int s_cnt[PLAN_MAX_E];
  __shared__ int s_off[PLAN_MAX_E];
  __shared__ int s_wr[PLAN_THREADS / 32], s_wt[PLAN_THREADS / 32];
  __shared__ int s_total;
  extern __shared__ int s_dyn[];    // PRIVATE: [PLAN_THREADS / 32][E] histograms; SMEM_ROWS: then row_of
  int* s_hist = s_dyn;
  int* s_rows = s_dyn + (PRIVATE ? (PLAN_THREADS / 32) * E : 0);
  int* rows_out = SMEM_ROWS ? s_rows : row_of;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  auto id_at = [&](int64_t i) { return ids[i]; };
  if (PRIVATE) {
    for (int k = tid; k < (PLAN_THREADS / 32) * E; k += PLAN_THREADS) s_hist[k] = 0;
  } else {
    for (int e = tid; e < E; e += PLAN_THREADS) s_cnt[e] = 0;
  }
  __syncthreads();
  for (int64_t i0 = tid; i0 < R; i0 += 4 * PLAN_THREADS) {
    int ev[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * PLAN_THREADS;
      ev[u] = i < R ? id_at(i) : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (ev[u] >= 0 && ev[u] < E) atomicAdd(PRIVATE ? &s_hist[wid * E + ev[u]] : &s_cnt[ev[u]], 1);
  }
  __syncthreads();
  if (PRIVATE) {
    for (int e = tid; e < E; e += PLAN_THREADS) {
      int run = 0;
      for (int w = 0; w < PLAN_THREADS / 32; ++w) {
        const int c = s_hist[w * E + e];
        s_hist[w * E + e] = run;
        run += c;
      }
      s_cnt[e] = run;
    }
    __syncthreads();
  }
  // block scan: thread tid owns experts [tid * ept, tid * ept + ept)
  const int ept = (E + PLAN_THREADS - 1) / PLAN_THREADS;
  int lr = 0, lt = 0;
  for (int j = 0; j < ept; ++j) {
    const int e = tid * ept + j;
    if (e < E) {
      lr += (s_cnt[e] + GV_MCHUNK - 1) / GV_MCHUNK * GV_MCHUNK;
      lt += (s_cnt[e] + tile_max - 1) / tile_max;
    }
  }
  int ir = lr, it = lt;   // inclusive within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ir, o), b = __shfl_up_sync(0xffffffffu, it, o);
    if (lane >= o) ir += a, it += b;
  }
  if (lane == 31) s_wr[wid] = ir, s_wt[wid] = it;
  __syncthreads();
  if (wid == 0) {
    int wr = s_wr[lane], wt = s_wt[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, wr, o), b = __shfl_up_sync(0xffffffffu, wt, o);
      if (lane >= o) wr += a, wt += b;
    }
    s_wr[lane] = wr, s_wt[lane] = wt;   // inclusive over warps
  }
  __syncthreads();
  int acc = (wid > 0 ? s_wr[wid - 1] : 0) + ir - lr;
  int tiles = (wid > 0 ? s_wt[wid - 1] : 0) + it - lt;
  for (int j = 0; j < ept; ++j) {
    const int e = tid * ept + j;
    if (e < E) {
      const int n = s_cnt[e];
      s_off[e] = acc;
      poff[e] = acc;
      // as many tiles as tile_max needs, of equal size rounded up to 32 rows
      // (at most tile_max, so there are exactly that many)
      const int nt = (n + tile_max - 1) / tile_max;
      const int sz = nt > 0 ? ((n + nt - 1) / nt + 31) / 32 * 32 : tile_max;
      for (int r = 0; r < n; r += sz, ++tiles) {
        tile_expert[tiles] = e;
        tile_row0[tiles] = acc + r;
        tile_rows[tiles] = min(sz, n - r);
      }
      for (int c = 0; c * GV_MCHUNK < n; ++c) {
        chunk_expert[acc / GV_MCHUNK + c] = e;
        chunk_rows[acc / GV_MCHUNK + c] = min(GV_MCHUNK, n - c * GV_MCHUNK);
      }
      acc += (n + GV_MCHUNK - 1) / GV_MCHUNK * GV_MCHUNK;
    }
  }
  if (tid == PLAN_THREADS - 1) {
    s_total = acc;
    *chunk_count = acc / GV_MCHUNK;
    *tile_count = tiles;
  }
  __syncthreads();
  for (int r = tid; r < s_total; r += PLAN_THREADS) rows_out[r] = -1;
  if (!PRIVATE)
    for (int e = tid; e < E; e += PLAN_THREADS) s_cnt[e] = 0;
  __syncthreads();   // row_of = -1 before any position is written; counts (or warp offsets) as cursors
  for (int64_t i0 = tid; i0 < R; i0 += 4 * PLAN_THREADS) {
    int ev[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * PLAN_THREADS;
      ev[u] = i < R ? id_at(i) : 0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * PLAN_THREADS;
      if (i >= R) continue;
      if (ev[u] < 0 || ev[u] >= E) {
        pos_of[i] = -1;
        atomicExch(status, NVFP4_ERR_INVALID_ARG);
        continue;
      }
      const int pos = s_off[ev[u]] + atomicAdd(PRIVATE ? &s_hist[wid * E + ev[u]] : &s_cnt[ev[u]], 1);
      rows_out[pos] = static_cast<int>(static_cast<uint32_t>(i) / static_cast<uint32_t>(topk));
      pos_of[i] = pos;
    }
  }
  if (SMEM_ROWS) {
    __syncthreads();
    for (int r = tid; r < s_total; r += PLAN_THREADS) row_of[r] = s_rows[r];
  }
}

// The routing plan over G CTAs of one cooperative launch (all resident), for
// many routed slots and E <= PLAN_COOP_MAX_E (the single-CTA plan spent ~20 us
// on 32,768 slots). CTA g counts the experts of its slice of the slots into
// hist[g][*]; after one grid barrier every CTA reads the whole count table,
// takes each expert's padded offset (block scan) and its own offset within
// each expert (the counts of the CTAs before it), and places its slots; CTA 0
// also writes the chunk and tile tables and marks each expert's padding rows
// with -1. The results are the single-CTA plan's up to the order of rows
// within an expert, which no output depends on. The barrier wait is bounded:
// a CTA that gives up records NVFP4_ERR_TIMEOUT and leaves.
__global__ void __launch_bounds__(PLAN_COOP_THREADS) route_plan_coop_kernel(
    const int32_t* ids, int64_t R, int topk, int E, int* poff, int* chunk_count, int* chunk_expert, int* chunk_rows,
    int* tile_count, int* tile_expert, int* tile_row0, int* tile_rows, int* row_of, int* pos_of, int* hist,
    unsigned int* bar, int* status, int tile_max) {
  __shared__ int s_cnt[PLAN_COOP_MAX_E];   // this CTA's counts, then its cursors
  __shared__ int s_off[PLAN_COOP_MAX_E];   // expert base + this CTA's offset within the expert
  __shared__ int s_tot[PLAN_COOP_MAX_E];
  __shared__ int s_pb[PLAN_COOP_THREADS], s_pt[PLAN_COOP_THREADS];   // partial sums [part][E]
  __shared__ int s_abort;
  const int tid = threadIdx.x, G = static_cast<int>(gridDim.x), g = static_cast<int>(blockIdx.x);
  const int64_t slice = (R + G - 1) / G;
  const int64_t i_begin = g * slice, i_end = i_begin + slice < R ? i_begin + slice : R;
  for (int e = tid; e < E; e += PLAN_COOP_THREADS) s_cnt[e] = 0;
  if (tid == 0) s_abort = 0;
  __syncthreads();
  for (int64_t i = i_begin + tid; i < i_end; i += PLAN_COOP_THREADS) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += PLAN_COOP_THREADS) hist[g * E + e] = s_cnt[e];
  // grid barrier: every CTA's counts are in hist
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 0; *reinterpret_cast<volatile unsigned int*>(bar) < static_cast<unsigned int>(G); ++n) {
      if ((n & 63) == 63 && globaltimer() - t0 > WAIT_LIMIT_NS) {
        atomicExch(status, NVFP4_ERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
  }
  __syncthreads();
  if (s_abort) return;
  // totals and this CTA's offset within each expert: `parts` threads per
  // expert, each summing every parts-th CTA's count (independent loads)
  const int parts = PLAN_COOP_THREADS / E;   // >= 2
  if (tid < parts * E) {
    const int e = tid % E, part = tid / E;
    int before = 0, tot = 0;
#pragma unroll 4
    for (int h = part; h < G; h += parts) {
      const int c = __ldcg(hist + h * E + e);
      before += h < g ? c : 0;
      tot += c;
    }
    s_pb[part * E + e] = before;
    s_pt[part * E + e] = tot;
  }
  __syncthreads();
  for (int e = tid; e < E; e += PLAN_COOP_THREADS) {
    int before = 0, tot = 0;
    for (int part = 0; part < parts; ++part) before += s_pb[part * E + e], tot += s_pt[part * E + e];
    s_tot[e] = tot;
    s_off[e] = before;
    s_cnt[e] = 0;
  }
  __syncthreads();
  // expert base offsets (padded to GV_MCHUNK rows): a scan by warp 0, E <= 256
  if (tid < 32) {
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + tid;
      const int pr = e < E ? (s_tot[e] + GV_MCHUNK - 1) / GV_MCHUNK * GV_MCHUNK : 0;
      int inc = pr;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, inc, o);
        if (tid >= o) inc += a;
      }
      if (e < E) {
        const int ex = base + inc - pr;   // exclusive
        s_off[e] += ex;
        if (g == 0) poff[e] = ex;
      }
      base += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (g == 0 && tid == 0) *chunk_count = base / GV_MCHUNK;
  }
  __syncthreads();
  if (g == 0) {
    // tables (one thread per expert; tile index from a scan of tile counts)
    if (tid < 32) {
      int tbase = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + tid;
        const int n = e < E ? s_tot[e] : 0;
        const int nt = (n + tile_max - 1) / tile_max;
        int inc = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int a = __shfl_up_sync(0xffffffffu, inc, o);
          if (tid >= o) inc += a;
        }
        if (e < E) {
          const int acc = s_off[e];   // CTA 0: its own offset within each expert is 0
          int tiles = tbase + inc - nt;
          const int sz = nt > 0 ? ((n + nt - 1) / nt + 31) / 32 * 32 : tile_max;
          for (int r = 0; r < n; r += sz, ++tiles) {
            tile_expert[tiles] = e;
            tile_row0[tiles] = acc + r;
            tile_rows[tiles] = min(sz, n - r);
          }
          for (int c = 0; c * GV_MCHUNK < n; ++c) {
            chunk_expert[acc / GV_MCHUNK + c] = e;
            chunk_rows[acc / GV_MCHUNK + c] = min(GV_MCHUNK, n - c * GV_MCHUNK);
          }
          // the expert's padding rows hold no token
          for (int r = n; r < (n + GV_MCHUNK - 1) / GV_MCHUNK * GV_MCHUNK; ++r) row_of[acc + r] = -1;
        }
        tbase += __shfl_sync(0xffffffffu, inc, 31);
      }
      if (tid == 0) *tile_count = tbase;
    }
  }
  // place this CTA's slots
  for (int64_t i = i_begin + tid; i < i_end; i += PLAN_COOP_THREADS) {
    const int e = ids[i];
    if (e < 0 || e >= E) {
      pos_of[i] = -1;
      atomicExch(status, NVFP4_ERR_INVALID_ARG);
      continue;
    }
    const int pos = s_off[e] + atomicAdd(&s_cnt[e], 1);
    row_of[pos] = static_cast<int>(static_cast<uint32_t>(i) / static_cast<uint32_t>(topk));
    pos_of[i] = pos;
  }
}

template <bool PRIVATE, bool SMEM_ROWS>
int launch_route_plan_t(const int32_t* ids, int64_t R, int topk, int64_t E, const MoeWs& m, int tile_max,
                        cudaStream_t stream) {
  const int64_t rows_max = R + GV_MCHUNK * E;   // the padded rows never exceed this
  const int smem =
      static_cast<int>(((PRIVATE ? (PLAN_THREADS / 32) * E : 0) + (SMEM_ROWS ? rows_max : 0)) * sizeof(int));
  auto k = route_plan_kernel<PRIVATE, SMEM_ROWS>;
  const int rc = ensure_smem(k, smem > 0 ? smem : 1);
  if (rc != NVFP4_OK) return rc;
  k<<<1, PLAN_THREADS, smem, stream>>>(ids, R, topk, static_cast<int>(E), m.poff, m.chunk_count, m.chunk_expert,
                                       m.chunk_rows, m.tile_count, m.tile_expert, m.tile_row0, m.tile_rows, m.row_of,
                                       m.pos_of, device_status_ptr(), tile_max);
  return from_cuda(cudaGetLastError());
}

// tile_max: a multiple of 32, at least PLAN_TILE_MIN
int launch_route_plan(const int32_t* ids, int64_t R, int topk, int64_t E, const MoeWs& m, int tile_max,
                      cudaStream_t stream) {
  if (E <= PLAN_COOP_MAX_E && R >= 16LL * PLAN_COOP_SLICE) {
    int64_t G = (R + PLAN_COOP_SLICE - 1) / PLAN_COOP_SLICE;
    const int64_t cap = sm_count() < PLAN_COOP_MAX_G ? sm_count() : PLAN_COOP_MAX_G;   // one CTA per SM fits
    if (G > cap) G = cap;
    if (cudaMemsetAsync(m.plan_bar, 0, sizeof(unsigned int), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(G));
    cfg.blockDim = dim3(PLAN_COOP_THREADS);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int* status = device_status_ptr();
    const int Ei = static_cast<int>(E);
    return from_cuda(cudaLaunchKernelEx(&cfg, route_plan_coop_kernel, ids, R, topk, Ei, m.poff, m.chunk_count,
                                        m.chunk_expert, m.chunk_rows, m.tile_count, m.tile_expert, m.tile_row0,
                                        m.tile_rows, m.row_of, m.pos_of, m.plan_hist, m.plan_bar, status, tile_max));
  }
  const bool priv = E <= PLAN_PRIVATE_MAX_E;
  const bool staged = R + GV_MCHUNK * E <= PLAN_SMEM_ROWS_MAX;
  if (priv && staged) return launch_route_plan_t<true, true>(ids, R, topk, E, m, tile_max, stream);
  if (priv) return launch_route_plan_t<true, false>(ids, R, topk, E, m, tile_max, stream);
  if (staged) return launch_route_plan_t<false, true>(ids, R, topk, E, m, tile_max, stream);
  return launch_route_plan_t<false, false>(ids, R, topk, E, m, tile_max, stream);
}

// One CTA per padded row (rows longer than MOE_PREP_MAX_K).
__global__ void __launch_bounds__(GV_THREADS) xprep_moe_row_kernel(const uint16_t* src, int64_t K, bool gather,
                                                                    const int* row_of, const int* chunk_count,
                                                                    uint4* xfrag, int* pexp) {
  const int64_t r = blockIdx.x;
  if (r >= static_cast<int64_t>(*chunk_count) * GV_MCHUNK) return;
  const int tok = row_of[r];
  const uint16_t* s = nullptr;
  if (tok >= 0) s = gather ? src + static_cast<int64_t>(tok) * K : src + r * K;
  xprep_row(s, K, r, xfrag, pexp);
}

// One warp per padded row: gather (tokens) or pass through (h), to
// fragments. The warp reads its row once into registers (CH 16-byte pieces
// per lane, K <= 256 * CH <= 4096), takes the amax with shuffles and converts
// (the same per-row shift and rounding as xprep_row).
constexpr int MOE_PREP_WARPS = 8;
constexpr int MOE_PREP_MAX_K = 4096;
template <int CH>
__global__ void __launch_bounds__(MOE_PREP_WARPS * 32) xprep_moe_kernel(const uint16_t* src, int64_t K, bool gather,
                                                                         const int* row_of, const int* chunk_count,
                                                                         uint4* xfrag, int* pexp) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * MOE_PREP_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= static_cast<int64_t>(*chunk_count) * GV_MCHUNK) return;
  const int tok = row_of[r];
  const uint16_t* s = nullptr;
  if (tok >= 0) s = gather ? src + static_cast<int64_t>(tok) * K : src + r * K;
  const int64_t n8 = K / 8;
  uint4 v[CH];
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int64_t q = lane + 32 * c;
    v[c] = make_uint4(0, 0, 0, 0);
    if (s != nullptr && q < n8) v[c] = __ldg(reinterpret_cast<const uint4*>(s) + q);
    const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w4[e] & 0xFFFFu)));
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w4[e] >> 16)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int p = 0;
  if (amax > 0.f) p = min(max(ilogbf(amax) - 14, -100), 113);
  const float mul = ldexpf(1.0f, -p);
  if (lane == 0) pexp[r] = p;
  const int64_t chunk = r / GV_MCHUNK;
  const int nt = static_cast<int>((r % GV_MCHUNK) / 8);
  const int g = static_cast<int>(r % 8);
  const int64_t n_it = K / GV_KIT;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int64_t q = lane + 32 * c;
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

// The same per-row conversion into row-major f16 rows [padded rows][K] (the
// tensor-core path's B operand, read by TMA): one warp per padded row, CH
// 16-byte pieces per lane (K <= 256 * CH), so short rows keep few registers.
template <int CH>
__global__ void __launch_bounds__(MOE_PREP_WARPS * 32) xprep_moe_rows_kernel(const uint16_t* src, int64_t K,
                                                                              bool gather, const int* row_of,
                                                                              const int* chunk_count, uint4* xrow,
                                                                              int* pexp) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * MOE_PREP_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= static_cast<int64_t>(*chunk_count) * GV_MCHUNK) return;
  const int tok = row_of[r];
  const uint16_t* s = nullptr;
  if (tok >= 0) s = gather ? src + static_cast<int64_t>(tok) * K : src + r * K;
  const int64_t n8 = K / 8;
  uint4 v[CH];
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int64_t q = lane + 32 * c;
    v[c] = make_uint4(0, 0, 0, 0);
    if (s != nullptr && q < n8) v[c] = __ldg(reinterpret_cast<const uint4*>(s) + q);
    const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w4[e] & 0xFFFFu)));
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w4[e] >> 16)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int p = 0;
  if (amax > 0.f) p = min(max(ilogbf(amax) - 14, -100), 113);
  const float mul = ldexpf(1.0f, -p);
  if (lane == 0) pexp[r] = p;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int64_t q = lane + 32 * c;
    if (q < n8) {
      uint4 o;
      o.x = f32x2_to_f16x2(bf16_bits_to_f32(v[c].x & 0xFFFFu) * mul, bf16_bits_to_f32(v[c].x >> 16) * mul);
      o.y = f32x2_to_f16x2(bf16_bits_to_f32(v[c].y & 0xFFFFu) * mul, bf16_bits_to_f32(v[c].y >> 16) * mul);
      o.z = f32x2_to_f16x2(bf16_bits_to_f32(v[c].z & 0xFFFFu) * mul, bf16_bits_to_f32(v[c].z >> 16) * mul);
      o.w = f32x2_to_f16x2(bf16_bits_to_f32(v[c].w & 0xFFFFu) * mul, bf16_bits_to_f32(v[c].w >> 16) * mul);
      xrow[r * n8 + q] = o;
    }
  }
}

// out[t][c] = bf16(sum_j w[t][j] * y[pos(t, j)][c]) in fp32, slots in order
// (y: the bf16 expert outputs); one thread per 4 columns (H % 4 == 0), CTA
// (t, column block of 1024).
__global__ void combine_kernel(const uint16_t* ybuf, const int* pos_of, const float* w, int64_t T, int topk,
                               int64_t H, uint16_t* out) {
  const int64_t t = blockIdx.x;
  const int64_t c = (static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x) * 4;
  if (c >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < topk; ++j) {
    const int pos = pos_of[t * topk + j];
    if (pos < 0) continue;
    const float wj = w[t * topk + j];
    const uint2 yb = *reinterpret_cast<const uint2*>(ybuf + static_cast<int64_t>(pos) * H + c);
    acc.x = fmaf(wj, bf16_bits_to_f32(yb.x & 0xFFFFu), acc.x);
    acc.y = fmaf(wj, bf16_bits_to_f32(yb.x >> 16), acc.y);
    acc.z = fmaf(wj, bf16_bits_to_f32(yb.y & 0xFFFFu), acc.z);
    acc.w = fmaf(wj, bf16_bits_to_f32(yb.y >> 16), acc.w);
  }
  uint2 o;
  o.x = f32_to_bf16_bits(acc.x) | (f32_to_bf16_bits(acc.y) << 16);
  o.y = f32_to_bf16_bits(acc.z) | (f32_to_bf16_bits(acc.w) << 16);
  *reinterpret_cast<uint2*>(out + t * H + c) = o;
}

// One expert GEMM on the TMA-fed skinny kernel: one CTA per (32-token chunk,
// row tile), CTAs of unused chunks exit at once. W is the stack of the E
// experts' matrices, viewed as one [E * rows][K] matrix; box_rows = 64 for
// gate/up (64 gate rows and the matching 64 up rows per tile), 128 for down.
template <int MODE>
int launch_moe_tma(const nvfp4_tensor_t& W, int box_rows, const TmaSkinnyParams& p, dim3 grid, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(W.batch) * W.rows;
  CUtensorMap mc, ms;
  int rc = make_tmap_2d_u8(&mc, W.codes, W.K / 2, rows, W.K / 2, 128, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != NVFP4_OK) return rc;
  rc = make_tmap_2d_u8(&ms, W.scales, W.K / 16, rows, W.K / 16, 16, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != NVFP4_OK) return rc;
  auto k = skinny_tma_kernel<4, MODE, 2, 2>;
  rc = ensure_smem(k, GtCfg<4>::SMEM);
  if (rc != NVFP4_OK) return rc;
  return launch_ex(k, grid, dim3(GtWarps<2, 2>::THREADS), GtCfg<4>::SMEM, 1, false, stream, mc, ms, p);
}

// Activation prep of the routed rows (K = H: gather tokens; K = I: pass h through).
int prep_moe(const uint16_t* src, int64_t K, bool gather, const MoeWs& m, uint4* xfrag, int* pexp,
             cudaStream_t stream) {
  const int64_t prow = m.max_chunks * GV_MCHUNK;
  const dim3 grid(static_cast<unsigned>(ceil_div(prow, MOE_PREP_WARPS))), block(MOE_PREP_WARPS * 32);
  if (K <= 1024)
    xprep_moe_kernel<4><<<grid, block, 0, stream>>>(src, K, gather, m.row_of, m.chunk_count, xfrag, pexp);
  else if (K <= 2048)
    xprep_moe_kernel<8><<<grid, block, 0, stream>>>(src, K, gather, m.row_of, m.chunk_count, xfrag, pexp);
  else if (K <= MOE_PREP_MAX_K)
    xprep_moe_kernel<16><<<grid, block, 0, stream>>>(src, K, gather, m.row_of, m.chunk_count, xfrag, pexp);
  else
    xprep_moe_row_kernel<<<static_cast<unsigned>(prow), GV_THREADS, 0, stream>>>(src, K, gather, m.row_of,
                                                                                  m.chunk_count, xfrag, pexp);
  return from_cuda(cudaGetLastError());
}

// Row-major f16 prep of the routed rows for the tensor-core path.
int prep_moe_rows(const uint16_t* src, int64_t K, bool gather, const MoeWs& m, void* xrow, int* pexp,
                  cudaStream_t stream) {
  const int64_t prow = m.max_chunks * GV_MCHUNK;
  const dim3 grid(static_cast<unsigned>(ceil_div(prow, MOE_PREP_WARPS))), block(MOE_PREP_WARPS * 32);
  uint4* dst = static_cast<uint4*>(xrow);
  if (K <= 1024)
    xprep_moe_rows_kernel<4><<<grid, block, 0, stream>>>(src, K, gather, m.row_of, m.chunk_count, dst, pexp);
  else if (K <= 2048)
    xprep_moe_rows_kernel<8><<<grid, block, 0, stream>>>(src, K, gather, m.row_of, m.chunk_count, dst, pexp);
  else
    xprep_moe_rows_kernel<16><<<grid, block, 0, stream>>>(src, K, gather, m.row_of, m.chunk_count, dst, pexp);
  return from_cuda(cudaGetLastError());
}

// One expert GEMM on the tensor cores: a persistent kernel, one CTA pair per
// two SMs walking the (tile, weight-block pair) items that the routing plan
// produced. xrow holds the f16 rows [padded rows][K].
template <bool GATEUP>
int launch_moe_tc(const nvfp4_tensor_t& W, const MoeWs& m, const void* xrow, const MoeTcParams& p,
                  cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(W.batch) * W.rows;
  const int64_t prow = m.max_chunks * GV_MCHUNK;
  CUtensorMap mx, mw;
  int rc = make_tmap_2d_u16(&mx, xrow, p.K, prow, static_cast<int64_t>(p.K) * 2, 64, XT_NMAX / 2,
                            CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != NVFP4_OK) return rc;
  // codes in 64-byte rows (128 K), 64B swizzle; gate/up: 64 gate rows and
  // the 64 up rows I further on in one box
  rc = GATEUP ? make_tmap_3d_u8(&mw, W.codes, W.K / 2, rows, 2, W.K / 2, static_cast<int64_t>(p.inter) * (W.K / 2), 64,
                                64, 2, CU_TENSOR_MAP_SWIZZLE_64B)
              : make_tmap_2d_u8(&mw, W.codes, W.K / 2, rows, W.K / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B);
  if (rc != NVFP4_OK) return rc;
  // the output: gate/up h [rows][I], boxes of 16 columns; down y [rows][H], 32 columns
  CUtensorMap mo;
  rc = GATEUP ? make_tmap_2d_u16(&mo, p.h_out, p.inter, prow, static_cast<int64_t>(p.inter) * 2, 16, 32,
                                 CU_TENSOR_MAP_SWIZZLE_NONE)
              : make_tmap_2d_u16(&mo, p.y_out, p.hidden, prow, static_cast<int64_t>(p.hidden) * 2, 32, 32,
                                 CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != NVFP4_OK) return rc;
  auto k = moe_tc_kernel<GATEUP>;
  rc = ensure_smem(k, XT_SMEM);
  if (rc != NVFP4_OK) return rc;
  const int64_t work_max = m.max_tiles * (GATEUP ? p.inter / 64 : p.hidden / 128) / 2;
  const int64_t pairs_max = sm_count() / 2;
  const unsigned grid = static_cast<unsigned>(2 * (work_max < pairs_max ? work_max : pairs_max));
  return launch_ex(k, dim3(grid), dim3(XT_THREADS), XT_SMEM, 2, false, stream, mx, mw, mo, p);
}

int combine(const MoeWs& m, const float* w, int64_t T, int topk, int64_t H, uint16_t* out, cudaStream_t stream) {
  combine_kernel<<<dim3(static_cast<unsigned>(T), static_cast<unsigned>(ceil_div(H, 1024))), 256, 0, stream>>>(
      m.ybuf, m.pos_of, w, T, topk, H, out);
  return from_cuda(cudaGetLastError());
}

}  // namespace

int launch_moe_route(const float* logits, int64_t T, int E, int topk, int32_t* ids, float* weights,
                     cudaStream_t stream) {
  if (T == 0) return NVFP4_OK;
  const int warps = 4;
  const unsigned grid = static_cast<unsigned>(ceil_div(T, warps));
  if (E <= 128)
    route_reg_kernel<4><<<grid, warps * 32, 0, stream>>>(logits, T, E, topk, ids, weights);
  else if (E <= 256)
    route_reg_kernel<8><<<grid, warps * 32, 0, stream>>>(logits, T, E, topk, ids, weights);
  else
    route_kernel<<<grid, warps * 32, 0, stream>>>(logits, T, E, topk, ids, weights);
  return from_cuda(cudaGetLastError());
}

size_t grouped_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk) {
  return carve_moe(nullptr, T, H, I, E, topk).bytes;
}

size_t grouped_w4a4_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk) {
  return carve_moe(nullptr, T, H, I, E, topk, true).bytes;
}

// The routed-expert layer with 4-bit activations (reading R10): the layer
// input quantised once with its own dynamic tensor scale and gathered per
// expert tile, the gate/up GEMM on the block-scaled FP4 tensor cores with
// SiLU * mul and the amax of h fused into its epilogue, every routed h row
// quantised with one dynamic tensor scale, the down GEMM, and the combine of
// the W4A16 layer (slots in order, deterministic).
int launch_grouped_gemm_w4a4(const uint16_t* X, int64_t T, int topk, const int32_t* ids, const float* w,
                             const nvfp4_tensor_t& W13, const nvfp4_tensor_t& W2, uint16_t* out, void* ws,
                             cudaStream_t stream) {
  if (T == 0) return NVFP4_OK;
  const int64_t E = W13.batch, I = W13.rows / 2, H = W13.K;
  const int64_t R = T * topk;
  if (E > PLAN_MAX_E || R >= (1LL << 31)) return NVFP4_ERR_UNSUPPORTED_SHAPE;   // plan positions are int
  const MoeWs m = carve_moe(ws, T, H, I, E, topk, true);
  // experts with 256+ routed rows on average: CTA pairs over 256-row tiles;
  // fewer: one CTA per 128-row tile (a pair's 256 rows would be mostly padding)
  const bool pair = R >= static_cast<int64_t>(W4A4_TILE) * E;
  const int tile = pair ? W4A4_TILE : PLAN_TILE_MIN;
  const int64_t trows = (ceil_div(R, tile) + E) * tile;   // <= w4a4_tile_rows(R, E), the buffers' rows
  if (trows >= (1LL << 31) / (H / 2)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  int rc = launch_route_plan(ids, R, topk, E, m, tile, stream);
  if (rc != NVFP4_OK) return rc;
  // the layer input quantised once per token (dynamic tensor scale), then its
  // routed rows gathered into the tile-major matrix
  rc = launch_quantize(X, NVFP4_DTYPE_BF16, T, H, m.xt_codes, m.xt_scales, m.st, NVFP4_ST_COMPUTE,
                       NVFP4_SCALES_ROWMAJOR, m.q_ws, stream);
  if (rc != NVFP4_OK) return rc;
  if (cudaMemsetAsync(m.amax + 1, 0, sizeof(unsigned int), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  const unsigned qgrid = static_cast<unsigned>(trows / QR_WARPS);
  gather_routed_kernel<<<qgrid, 8 * 32, 0, stream>>>(m.xt_codes, m.xt_scales, H, m.row_of, m.tile_count, m.tile_row0,
                                                     m.tile_rows, m.xq_codes, m.xq_scales, tile);
  rc = from_cuda(cudaGetLastError());
  if (rc != NVFP4_OK) return rc;
  rc = launch_grouped_w4a4(true, m.xq_codes, m.xq_scales, m.st, trows, W13, m.tile_count, m.tile_expert, m.tile_row0,
                           m.tile_rows, m.max_tiles, static_cast<int>(I), static_cast<int>(H), m.hbuf, m.amax + 1,
                           nullptr, m.max_chunks * GV_MCHUNK, pair, stream);
  if (rc != NVFP4_OK) return rc;
  quantize_routed_kernel<<<qgrid, QR_WARPS * 32, 0, stream>>>(m.hbuf, I, false, m.row_of, m.tile_count, m.tile_row0,
                                                              m.tile_rows, m.amax + 1, m.st + 1, m.hq_codes,
                                                              m.hq_scales, tile);
  rc = from_cuda(cudaGetLastError());
  if (rc != NVFP4_OK) return rc;
  rc = launch_grouped_w4a4(false, m.hq_codes, m.hq_scales, m.st + 1, trows, W2, m.tile_count, m.tile_expert,
                           m.tile_row0, m.tile_rows, m.max_tiles, static_cast<int>(I), static_cast<int>(H), nullptr,
                           nullptr, m.ybuf, m.max_chunks * GV_MCHUNK, pair, stream);
  if (rc != NVFP4_OK) return rc;
  return combine(m, w, T, topk, H, out, stream);
}

int launch_grouped_gemm(const uint16_t* X, int64_t T, int topk, const int32_t* ids, const float* w,
                        const nvfp4_tensor_t& W13, const nvfp4_tensor_t& W2, uint16_t* out, void* ws,
                        cudaStream_t stream) {
  if (T == 0) return NVFP4_OK;
  const int64_t E = W13.batch, I = W13.rows / 2, H = W13.K;
  const int64_t R = T * topk;
  if (E > PLAN_MAX_E || R >= (1LL << 31)) return NVFP4_ERR_UNSUPPORTED_SHAPE;   // plan positions are int
  const MoeWs m = carve_moe(ws, T, H, I, E, topk);
  int rc = launch_route_plan(ids, R, topk, E, m, XT_NMAX, stream);
  if (rc != NVFP4_OK) return rc;

  // Many rows per expert: the tensor cores (the f16 rows live where the
  // fragment-order copies would).
  if (R >= XT_MIN_ROWS_PER_EXPERT * E && m.max_tiles <= 65535 && H % 256 == 0 && I % 256 == 0 && H <= MOE_PREP_MAX_K &&
      I <= MOE_PREP_MAX_K && ((reinterpret_cast<uintptr_t>(W13.scales) | reinterpret_cast<uintptr_t>(W2.scales)) & 15) == 0) {
    rc = prep_moe_rows(X, H, true, m, m.xfrag1, m.pexp1, stream);
    if (rc != NVFP4_OK) return rc;
    MoeTcParams p{};
    p.scales = W13.scales;
    p.s_t = W13.s_t;
    p.pexp = m.pexp1;
    p.tile_count = m.tile_count;
    p.tile_expert = m.tile_expert;
    p.tile_row0 = m.tile_row0;
    p.tile_rows = m.tile_rows;
    p.K = static_cast<int>(H);
    p.rows_per_expert = static_cast<int>(2 * I);
    p.inter = static_cast<int>(I);
    p.hidden = static_cast<int>(H);
    p.h_out = m.hbuf;
    p.status = device_status_ptr();
    rc = launch_moe_tc<true>(W13, m, m.xfrag1, p, stream);
    if (rc != NVFP4_OK) return rc;
    rc = prep_moe_rows(m.hbuf, I, false, m, m.xfrag2, m.pexp2, stream);
    if (rc != NVFP4_OK) return rc;
    MoeTcParams q = p;
    q.scales = W2.scales;
    q.s_t = W2.s_t;
    q.pexp = m.pexp2;
    q.K = static_cast<int>(I);
    q.rows_per_expert = static_cast<int>(H);
    q.h_out = nullptr;
    q.y_out = m.ybuf;
    rc = launch_moe_tc<false>(W2, m, m.xfrag2, q, stream);
    if (rc != NVFP4_OK) return rc;
    return combine(m, w, T, topk, H, out, stream);
  }

  rc = prep_moe(X, H, true, m, m.xfrag1, m.pexp1, stream);
  if (rc != NVFP4_OK) return rc;

  if (H % 256 == 0 && I % 256 == 0) {
    TmaSkinnyParams p{};
    p.s_t = W13.s_t;
    p.K = H;
    p.xfrag = m.xfrag1;
    p.pexp = m.pexp1;
    p.split = 1;
    p.chunk_count = m.chunk_count;
    p.chunk_expert = m.chunk_expert;
    p.chunk_rows = m.chunk_rows;
    p.inter = I;
    p.hidden = H;
    p.rows_per_expert = 2 * I;
    p.h_out = m.hbuf;
    p.status = device_status_ptr();
    p.weights_once = R <= GV_MCHUNK * E;   // about one token chunk per expert
    rc = launch_moe_tma<SK_MOE_GATEUP>(W13, 64, p,
                                       dim3(static_cast<unsigned>(m.max_chunks), static_cast<unsigned>(I / 64)),
                                       stream);
    if (rc != NVFP4_OK) return rc;
    rc = prep_moe(m.hbuf, I, false, m, m.xfrag2, m.pexp2, stream);
    if (rc != NVFP4_OK) return rc;
    TmaSkinnyParams q = p;
    q.s_t = W2.s_t;
    q.K = I;
    q.xfrag = m.xfrag2;
    q.pexp = m.pexp2;
    q.rows_per_expert = H;
    q.h_out = nullptr;
    q.y_out = m.ybuf;
    rc = launch_moe_tma<SK_MOE_DOWN>(
        W2, 128, q, dim3(static_cast<unsigned>(m.max_chunks), static_cast<unsigned>(ceil_div(H, GV_ROWS))), stream);
    if (rc != NVFP4_OK) return rc;
    return combine(m, w, T, topk, H, out, stream);
  }

  SkinnyParams p{};
  p.codes = W13.codes;
  p.scales = W13.scales;
  p.s_t = W13.s_t;
  p.K = H;
  p.xfrag = m.xfrag1;
  p.pexp = m.pexp1;
  p.split = 1;
  p.chunk_count = m.chunk_count;
  p.chunk_expert = m.chunk_expert;
  p.chunk_rows = m.chunk_rows;
  p.inter = I;
  p.hidden = H;
  p.rows_per_expert = 2 * I;
  p.h_out = m.hbuf;
  rc = launch_cluster(skinny_kernel<4, SK_MOE_GATEUP>,
                      dim3(static_cast<unsigned>(m.max_chunks), static_cast<unsigned>(I / 64)), dim3(GV_THREADS),
                      0, 1, stream, p);
  if (rc != NVFP4_OK) return rc;

  rc = prep_moe(m.hbuf, I, false, m, m.xfrag2, m.pexp2, stream);
  if (rc != NVFP4_OK) return rc;

  SkinnyParams q = p;
  q.codes = W2.codes;
  q.scales = W2.scales;
  q.s_t = W2.s_t;
  q.K = I;
  q.xfrag = m.xfrag2;
  q.pexp = m.pexp2;
  q.rows_per_expert = H;
  q.h_out = nullptr;
  q.y_out = m.ybuf;
  rc = launch_cluster(skinny_kernel<4, SK_MOE_DOWN>,
                      dim3(static_cast<unsigned>(m.max_chunks), static_cast<unsigned>(ceil_div(H, GV_ROWS))),
                      dim3(GV_THREADS), 0, 1, stream, q);
  if (rc != NVFP4_OK) return rc;

  return combine(m, w, T, topk, H, out, stream);
}

}  // namespace nvfp4
