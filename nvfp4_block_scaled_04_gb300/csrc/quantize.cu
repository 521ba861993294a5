// NVFP4 quantiser: amax pass (tensor scale) and the per-16 block quantiser,
// plus the re-layout of row-major block scales into the MMA scale layout.
//
// Every decision is taken in fp32 with IEEE division and multiplication
// (__fdiv_rn / __fmul_rn, no contraction into FMA):
//   s_t   = amax / 2688           (1 if amax == 0; or given)
//   sb    = amax_block / (s_t * 6) -> E4M3, nearest even, saturating at 448
//   q     = x / (e4m3(sb) * s_t)   -> e2m1, nearest even, saturating at 6
// with the sign bit of x kept on codes whose magnitude rounds to zero, and a
// zero block scale forcing zero codes. Format: 4-bit e2m1 values with one
// 8-bit float scale per 16 elements (Serving Qwen3.8-27B in 4-bit with a
// masked speculative decoding head, "What the artifact is").
#include "common.cuh"
#include "launch.h"
#include "quant_core.cuh"
#include "tc_util.cuh"

namespace nvfp4 {

namespace {

constexpr int Q_THREADS = 256;

template <typename T>
NVFP4_DEV void load8(const T* p, float (&v)[8]);

template <>
NVFP4_DEV void load8<uint16_t>(const uint16_t* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = bf16_bits_to_f32(w[e] & 0xFFFFu);
    v[2 * e + 1] = bf16_bits_to_f32(w[e] >> 16);
  }
}

template <>
NVFP4_DEV void load8<float>(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// 16-byte load kept in L2 with the given policy (the quantise pass reads the
// same bytes again right after the amax pass).
NVFP4_DEV uint4 ld_hint_v4(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
template <typename T>
NVFP4_DEV void load8_keep(const T* p, float (&v)[8], uint64_t policy);
template <>
NVFP4_DEV void load8_keep<uint16_t>(const uint16_t* p, float (&v)[8], uint64_t policy) {
  const uint4 u = ld_hint_v4(p, policy);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = bf16_bits_to_f32(w[e] & 0xFFFFu);
    v[2 * e + 1] = bf16_bits_to_f32(w[e] >> 16);
  }
}
template <>
NVFP4_DEV void load8_keep<float>(const float* p, float (&v)[8], uint64_t policy) {
  const uint4 a = ld_hint_v4(p, policy), b = ld_hint_v4(p + 4, policy);
  v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
  v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}

// The amax pass: CTA b writes the largest |x| of its share to partial[b]
// (fp32 bits; non-negative floats order like their bit patterns), so nothing
// has to be zeroed before it; with ATOMIC, every CTA folds its maximum into
// partial[0] instead (zeroed by the caller). Four 8-element loads in flight per thread, kept
// in L2 (evict-last) for the quantise pass; the pass walks the tensor from
// its start to its end. The quantise pass is launched as its programmatic
// dependent: it may start (and load its first blocks) once every CTA of
// this pass has started.
template <typename T, bool ATOMIC = false>
__global__ void __launch_bounds__(Q_THREADS) amax_kernel(const T* x, int64_t n8, unsigned int* partial) {
  __shared__ float red[Q_THREADS / 32];
  pdl_launch_dependents();
  uint64_t keep;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
  float m = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    float v[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) load8_keep<T>(x + (i + u * stride) * 8, v[u], keep);
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[u][e]));
  }
  for (; i < n8; i += stride) {
    float v[8];
    load8_keep<T>(x + i * 8, v, keep);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
    for (int w = 0; w < Q_THREADS / 32; ++w) b = fmaxf(b, red[w]);
    if (ATOMIC) atomicMax(partial, __float_as_uint(b));
    else partial[blockIdx.x] = __float_as_uint(b);
  }
}

// 16-byte words of one 16-element block: 2 (bf16) or 4 (fp32).
template <typename T>
struct BlockWords {
  static constexpr int N = static_cast<int>(sizeof(T));
};

template <typename T>
NVFP4_DEV void unpack16(const uint4 (&w)[BlockWords<T>::N], float (&v)[16]);
template <>
NVFP4_DEV void unpack16<uint16_t>(const uint4 (&w)[2], float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t u[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * i + 2 * e] = __uint_as_float(u[e] << 16);
      v[8 * i + 2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
    }
  }
}
template <>
NVFP4_DEV void unpack16<float>(const uint4 (&w)[4], float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[4 * i] = __uint_as_float(w[i].x);
    v[4 * i + 1] = __uint_as_float(w[i].y);
    v[4 * i + 2] = __uint_as_float(w[i].z);
    v[4 * i + 3] = __uint_as_float(w[i].w);
  }
}

// Largest |x| of a block: bf16 words by packed abs-max (the magnitudes' order
// is exact in bf16), fp32 values by fmax.
template <typename T>
NVFP4_DEV float block_amax(const uint4 (&w)[BlockWords<T>::N], const float (&v)[16]);
template <>
NVFP4_DEV float block_amax<uint16_t>(const uint4 (&w)[2], const float (&)[16]) {
  const uint32_t u[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
  uint32_t m = u[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(u[i]));
  // each step takes the magnitudes of both inputs, so m holds max |u| per half
  return fmaxf(__uint_as_float((m & 0x7FFFu) << 16), __uint_as_float(m & 0x7FFF0000u));
}
template <>
NVFP4_DEV float block_amax<float>(const uint4 (&)[4], const float (&v)[16]) {
  float ab = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) ab = fmaxf(ab, fabsf(v[e]));
  return ab;
}

// One thread quantises BPT blocks of 16 elements, 32 blocks apart in the row:
// the raw words of all of them are requested before any is converted. A warp
// covers a chunk of 32 * BPT consecutive blocks of a row; warps take chunks
// from the END of the tensor backwards (right after the amax pass, the tail
// of the input is still in L2), stepping by the warp count without a division
// per step. MMA-layout scale offsets split into a row part (per chunk) and a
// column part: byte (row, col) of the layout with `cols4` (padded K/16)
// columns is tile * 512 + (row % 32) * 16 + ((row / 32) % 4) * 4 + col % 4,
// tile = (row / 128) * (cols4 / 4) + col / 4.
//
// Tensor scale: GIVEN reads *s_t; COMPUTE takes s_t = amax / 2688 (1 if amax
// is 0) with amax the largest of amax_bits[0 .. n_amax) (the amax pass's
// per-CTA maxima, or one value). In COMPUTE the kernel may run as the amax
// pass's programmatic dependent: its first blocks are loaded before it waits
// for that pass's results.
template <typename T, int LAYOUT>
__global__ void __launch_bounds__(Q_THREADS, 4) quantize_kernel(const T* x, int64_t rows, int64_t K,
                                                                 uint8_t* codes, uint8_t* scales,
                                                                 const unsigned int* amax_bits, int n_amax,
                                                                 float* s_t, int mode, int64_t cols4) {
  constexpr int NW = BlockWords<T>::N;
  constexpr int BPT = 4 / NW;   // 2 blocks (bf16) or 1 (fp32) per thread
  __shared__ unsigned int s_amax;
  __shared__ QuantTables s_tab;
  // chunk indices fit in 32 bits (checked at launch)
  const uint32_t bpr = static_cast<uint32_t>(K / 16);
  const int cpr = static_cast<int>((bpr + 32 * BPT - 1) / (32 * BPT));
  const int lane = threadIdx.x & 31;
  const int warps = static_cast<int>(gridDim.x * (blockDim.x / 32));
  const int n_chunks = static_cast<int>(rows * cpr);
  const int c0 = n_chunks - 1 - static_cast<int>(blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5));
  int row = c0 >= 0 ? c0 / cpr : -1, cc = c0 >= 0 ? c0 - row * cpr : 0;
  const int drow = warps / cpr, dcc = warps - drow * cpr;
  const int64_t tiles_per_row = cols4 >> 2;
  // two chunks in flight per warp: the next chunk's words are requested
  // before the current one is converted
  uint4 raw[BPT][NW], nxt[BPT][NW];
  auto load_chunk = [&](int r, int c, uint4 (&dst)[BPT][NW]) {
    const uint32_t b0 = static_cast<uint32_t>(c) * (32 * BPT) + lane;
    const T* xrow = x + static_cast<int64_t>(r) * K;
#pragma unroll
    for (int u = 0; u < BPT; ++u) {
      const uint32_t bi = b0 + 32 * u;
      const uint4* src = reinterpret_cast<const uint4*>(xrow + static_cast<int64_t>(bi < bpr ? bi : 0) * 16);
#pragma unroll
      for (int i = 0; i < NW; ++i) dst[u][i] = __ldg(src + i);
    }
  };
  // the chunk after (row, cc) in this warp's walk
  auto advance = [&](int& r, int& c) {
    c -= dcc;
    r -= drow;
    if (c < 0) {
      c += cpr;
      r -= 1;
    }
  };
  if (row >= 0) load_chunk(row, cc, raw);
  float st;
  if (mode == NVFP4_ST_COMPUTE) {
    pdl_wait();   // the amax pass's maxima are complete and visible
    if (threadIdx.x == 0) s_amax = 0u;
    __syncthreads();
    unsigned int m = 0u;
    for (int i = threadIdx.x; i < n_amax; i += blockDim.x) m = max(m, __ldcg(amax_bits + i));
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane == 0) atomicMax(&s_amax, m);
    __syncthreads();
    const float amax = __uint_as_float(s_amax);
    st = amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *s_t = st;
  } else {
    st = *s_t;
  }
  const float d = __fmul_rn(st, 6.0f);
  float rdh, rdl;
  recip_brackets(d, rdh, rdl);
  quant_tables_init(s_tab, st);
  __syncthreads();
  while (row >= 0) {
    int nrow = row, ncc = cc;
    advance(nrow, ncc);
    if (nrow >= 0) load_chunk(nrow, ncc, nxt);
    const uint32_t b0 = static_cast<uint32_t>(cc) * (32 * BPT) + lane;
    const int64_t srow = LAYOUT == NVFP4_SCALES_MMA
                             ? (static_cast<int64_t>(row >> 7) * tiles_per_row) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4
                             : static_cast<int64_t>(row) * bpr;
#pragma unroll
    for (int u = 0; u < BPT; ++u) {
      const uint32_t bi = b0 + 32 * u;
      if (bi >= bpr) continue;
      float v[16];
      unpack16<T>(raw[u], v);
      uint2 packed;
      const uint32_t sc = quant_block16_tab(v, block_amax<T>(raw[u], v), d, rdh, rdl, s_tab, packed);
      reinterpret_cast<uint2*>(codes)[static_cast<int64_t>(row) * bpr + bi] = packed;
      scales[LAYOUT == NVFP4_SCALES_MMA ? srow + (bi >> 2) * 512 + (bi & 3) : srow + bi] = static_cast<uint8_t>(sc);
    }
    row = nrow;
    cc = ncc;
#pragma unroll
    for (int u = 0; u < BPT; ++u)
#pragma unroll
      for (int i = 0; i < NW; ++i) raw[u][i] = nxt[u][i];
  }
}

__global__ void prepack_kernel(const uint8_t* src, int64_t batch, int64_t rows, int64_t K, uint8_t* dst,
                               int64_t rows_p, int64_t cols4) {
  const int64_t per = rows_p * cols4;
  const int64_t total = batch * per;
  const int64_t kc = K / 16;
  for (int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < total;
       o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = o / per, rem = o % per;
    const int64_t tile = rem >> 9, within = rem & 511;
    const int64_t rt = tile / (cols4 >> 2), ct = tile % (cols4 >> 2);
    const int64_t row = rt * 128 + ((within & 15) >> 2) * 32 + (within >> 4);
    const int64_t col = ct * 4 + (within & 3);
    dst[o] = (row < rows && col < kc) ? src[(b * rows + row) * kc + col] : static_cast<uint8_t>(0);
  }
}

int grid_for(int64_t work, int threads) {
  int64_t g = (work + threads - 1) / threads;
  const int64_t cap = 8LL * sm_count();
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

// the amax pass's per-CTA maxima: at most AMAX_MAX_CTAS of them
constexpr int AMAX_MAX_CTAS = 2048;
size_t quantize_workspace_bytes() { return AMAX_MAX_CTAS * sizeof(unsigned int); }

int launch_quantize(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                    float* s_t, int s_t_mode, int scale_layout, void* workspace, cudaStream_t stream) {
  unsigned int* amax = static_cast<unsigned int*>(workspace);
  const int64_t n8 = rows * K / 8;
  const int64_t cols4 = mma_scale_cols(K);
  if (scale_layout == NVFP4_SCALES_MMA && rows > 0 && (rows % 128 != 0 || cols4 != K / 16)) {
    const size_t bytes = static_cast<size_t>(mma_scale_rows(rows) * cols4);
    if (cudaMemsetAsync(scales, 0, bytes, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  int n_amax = 0;
  if (s_t_mode == NVFP4_ST_COMPUTE) {
    n_amax = grid_for(n8 > 0 ? n8 : 1, Q_THREADS);
    if (n_amax > AMAX_MAX_CTAS) n_amax = AMAX_MAX_CTAS;
    if (x_dtype == NVFP4_DTYPE_BF16)
      amax_kernel<uint16_t><<<n_amax, Q_THREADS, 0, stream>>>(static_cast<const uint16_t*>(x), n8, amax);
    else
      amax_kernel<float><<<n_amax, Q_THREADS, 0, stream>>>(static_cast<const float*>(x), n8, amax);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  if (rows * ((K / 16 + 63) / 64) >= (1LL << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  // one full wave of resident blocks (the chunks are walked with a grid
  // stride): a grid of 8 blocks per SM at 6 resident left a quarter of the
  // work to a second, partial wave
  const int g_max = grid_for(n8 > 0 ? n8 : 1, Q_THREADS);
  int rc = NVFP4_OK;
#define NVFP4_Q(T, L)                                                                                         \
  do {                                                                                                        \
    int per_sm = 0;                                                                                           \
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_kernel<T, L>, Q_THREADS, 0) !=        \
            cudaSuccess ||                                                                                    \
        per_sm < 1)                                                                                           \
      per_sm = 1;                                                                                             \
    const int g = g_max < per_sm * sm_count() ? g_max : per_sm * sm_count();                                  \
    rc = launch_ex(quantize_kernel<T, L>, dim3(g), dim3(Q_THREADS), 0, 1, s_t_mode == NVFP4_ST_COMPUTE, stream,  \
                   static_cast<const T*>(x), rows, K, codes, scales, static_cast<const unsigned int*>(amax),    \
                   n_amax, s_t, s_t_mode, cols4);                                                             \
  } while (0)
  if (x_dtype == NVFP4_DTYPE_BF16) {
    if (scale_layout == NVFP4_SCALES_MMA) NVFP4_Q(uint16_t, NVFP4_SCALES_MMA);
    else NVFP4_Q(uint16_t, NVFP4_SCALES_ROWMAJOR);
  } else {
    if (scale_layout == NVFP4_SCALES_MMA) NVFP4_Q(float, NVFP4_SCALES_MMA);
    else NVFP4_Q(float, NVFP4_SCALES_ROWMAJOR);
  }
#undef NVFP4_Q
  return rc;
}

int launch_amax_bf16(const uint16_t* x, int64_t n, unsigned int* amax_bits, cudaStream_t stream) {
  if (cudaMemsetAsync(amax_bits, 0, sizeof(unsigned int), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  const int64_t n8 = n / 8;
  if (n8 > 0) amax_kernel<uint16_t, true><<<grid_for(n8, Q_THREADS), Q_THREADS, 0, stream>>>(x, n8, amax_bits);
  return from_cuda(cudaGetLastError());
}

int launch_quantize_bf16_from_amax(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                                   const unsigned int* amax_bits, float* s_t, cudaStream_t stream) {
  const int64_t cols4 = mma_scale_cols(K);
  if (rows == 0) return NVFP4_OK;
  if (rows % 128 != 0 || cols4 != K / 16) {
    const size_t bytes = static_cast<size_t>(mma_scale_rows(rows) * cols4);
    if (cudaMemsetAsync(scales, 0, bytes, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  if (rows * ((K / 16 + 63) / 64) >= (1LL << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  auto k = quantize_kernel<uint16_t, NVFP4_SCALES_MMA>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, Q_THREADS, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
  const int g_max = grid_for(rows * K / 8, Q_THREADS);
  const int g = g_max < per_sm * sm_count() ? g_max : per_sm * sm_count();
  k<<<g, Q_THREADS, 0, stream>>>(x, rows, K, codes, scales, amax_bits, 1, s_t, NVFP4_ST_COMPUTE, cols4);
  return from_cuda(cudaGetLastError());
}

int launch_prepack_scales(const uint8_t* src, int64_t batch, int64_t rows, int64_t K, uint8_t* dst,
                          cudaStream_t stream) {
  const int64_t rows_p = mma_scale_rows(rows), cols4 = mma_scale_cols(K);
  const int64_t total = batch * rows_p * cols4;
  if (total == 0) return NVFP4_OK;
  prepack_kernel<<<grid_for(total, 256), 256, 0, stream>>>(src, batch, rows, K, dst, rows_p, cols4);
  return from_cuda(cudaGetLastError());
}

}  // namespace nvfp4
