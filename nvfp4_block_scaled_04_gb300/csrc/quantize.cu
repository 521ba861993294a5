// NVFP4 quantiser: amax pass (tensor scale) and the per-16 block quantiser,
// plus the re-layout of row-major block scales into the MMA scale layout.
//
// Every decision is taken in fp32 with IEEE division and multiplication
// (__fdiv_rn / __fmul_rn, no contraction into FMA):
//   s_t   = amax / 2688           (1 if amax == 0; or given)
//   sb    = amax_block / (s_t * 6) -> E4M3, nearest even, saturating at 448
//   q     = x / (e4m3(sb) * s_t)   -> e2m1, nearest even, saturating at 6
// with the sign bit of x kept on codes whose magnitude rounds to zero, and a
// zero block scale forcing zero codes. Format: "NVFP4 is 4-bit e2m1 with
// per-16 FP8 scales" (Serving Qwen3.8-27B in 4-bit with a masked speculative
// decoding head, "What the artifact is").
#include "common.cuh"
#include "launch.h"

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

template <typename T>
__global__ void __launch_bounds__(Q_THREADS) amax_kernel(const T* x, int64_t n8, unsigned int* out) {
  __shared__ float red[Q_THREADS / 32];
  float m = 0.f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float v[8];
    load8<T>(x + i * 8, v);
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
    // non-negative floats order like their bit patterns
    atomicMax(out, __float_as_uint(b));
  }
}

// Byte offset of block scale (row, col) in the MMA layout with `cols4`
// (padded K/16) columns.
NVFP4_DEV int64_t mma_scale_offset(int64_t row, int64_t col, int64_t cols4) {
  const int64_t tile = (row >> 7) * (cols4 >> 2) + (col >> 2);
  return tile * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (col & 3);
}

// Each lane quantises half a block (8 elements); lanes 2i and 2i+1 hold the
// two halves of one block.
template <typename T, int LAYOUT>
__global__ void __launch_bounds__(Q_THREADS) quantize_kernel(const T* x, int64_t rows, int64_t K,
                                                              uint8_t* codes, uint8_t* scales,
                                                              const unsigned int* amax_bits, float* s_t,
                                                              int mode, int64_t cols4) {
  float st;
  if (mode == NVFP4_ST_COMPUTE) {
    const float amax = __uint_as_float(*amax_bits);
    st = amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *s_t = st;
  } else {
    st = *s_t;
  }
  const float d = __fmul_rn(st, 6.0f);
  const int64_t halves_per_row = K / 8;
  const int64_t total = rows * halves_per_row;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < total;
       base += stride) {
    const int64_t h = base + lane;
    const bool valid = h < total;
    float v[8];
    if (valid) {
      load8<T>(x + h * 8, v);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = 0.f;
    }
    float am = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(v[e]));
    const float ab = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    const uint32_t sc = f32_to_e4m3(__fdiv_rn(ab, d));
    uint32_t packed = 0;
    if (sc != 0) {
      const float den = __fmul_rn(e4m3_to_f32(sc), st);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float q0 = __fdiv_rn(v[2 * e], den);
        const float q1 = __fdiv_rn(v[2 * e + 1], den);
        uint32_t byte = f32x2_to_e2m1x2(fabsf(q0), fabsf(q1));
        byte |= (__float_as_uint(v[2 * e]) >> 31) << 3;
        byte |= (__float_as_uint(v[2 * e + 1]) >> 31) << 7;
        packed |= byte << (8 * e);
      }
    }
    if (valid) {
      reinterpret_cast<uint32_t*>(codes)[h] = packed;
      if ((h & 1) == 0) {
        const int64_t row = h / halves_per_row;
        const int64_t col = (h % halves_per_row) >> 1;
        const int64_t off = LAYOUT == NVFP4_SCALES_MMA ? mma_scale_offset(row, col, cols4) : row * (K / 16) + col;
        scales[off] = static_cast<uint8_t>(sc);
      }
    }
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

size_t quantize_workspace_bytes() { return 256; }

int launch_quantize(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                    float* s_t, int s_t_mode, int scale_layout, void* workspace, cudaStream_t stream) {
  unsigned int* amax = static_cast<unsigned int*>(workspace);
  const int64_t n8 = rows * K / 8;
  const int64_t cols4 = mma_scale_cols(K);
  if (scale_layout == NVFP4_SCALES_MMA && rows > 0 && (rows % 128 != 0 || cols4 != K / 16)) {
    const size_t bytes = static_cast<size_t>(mma_scale_rows(rows) * cols4);
    if (cudaMemsetAsync(scales, 0, bytes, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  if (s_t_mode == NVFP4_ST_COMPUTE) {
    if (cudaMemsetAsync(amax, 0, sizeof(unsigned int), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (n8 > 0) {
      const int g = grid_for(n8, Q_THREADS);
      if (x_dtype == NVFP4_DTYPE_BF16)
        amax_kernel<uint16_t><<<g, Q_THREADS, 0, stream>>>(static_cast<const uint16_t*>(x), n8, amax);
      else
        amax_kernel<float><<<g, Q_THREADS, 0, stream>>>(static_cast<const float*>(x), n8, amax);
    }
  }
  const int g = grid_for(n8 > 0 ? n8 : 1, Q_THREADS);
#define NVFP4_Q(T, L)                                                                                  \
  quantize_kernel<T, L><<<g, Q_THREADS, 0, stream>>>(static_cast<const T*>(x), rows, K, codes, scales, \
                                                     amax, s_t, s_t_mode, cols4)
  if (x_dtype == NVFP4_DTYPE_BF16) {
    if (scale_layout == NVFP4_SCALES_MMA) NVFP4_Q(uint16_t, NVFP4_SCALES_MMA);
    else NVFP4_Q(uint16_t, NVFP4_SCALES_ROWMAJOR);
  } else {
    if (scale_layout == NVFP4_SCALES_MMA) NVFP4_Q(float, NVFP4_SCALES_MMA);
    else NVFP4_Q(float, NVFP4_SCALES_ROWMAJOR);
  }
#undef NVFP4_Q
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
