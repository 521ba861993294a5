// Host-side launch helpers and the internal interface between the C ABI
// (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

inline int from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

// Number of SMs of the current device (queried once per device).
int sm_count();

// Launch `kernel` with a thread-block cluster of `cluster_x` CTAs along x
// (plain launch when cluster_x == 1) and, with `pdl`, programmatic stream
// serialisation: the kernel may start while the previous kernel on the
// stream finishes, and must `griddepcontrol.wait` before reading its output.
template <typename Kernel, typename... Args>
int launch_ex(Kernel kernel, dim3 grid, dim3 block, size_t smem, int cluster_x, bool pdl, cudaStream_t stream,
              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return from_cuda(cudaLaunchKernelEx(&cfg, kernel, args...));
}

template <typename Kernel, typename... Args>
int launch_cluster(Kernel kernel, dim3 grid, dim3 block, size_t smem, int cluster_x, cudaStream_t stream,
                   Args... args) {
  return launch_ex(kernel, grid, block, smem, cluster_x, false, stream, args...);
}

// Raise a kernel's dynamic shared memory limit (once per kernel and device).
int ensure_smem_impl(const void* func, int bytes);
template <typename Kernel>
int ensure_smem(Kernel kernel, int bytes) {
  return ensure_smem_impl(reinterpret_cast<const void*>(kernel), bytes);
}

// ---- tma_host.cu: 2-D uint8 tensor map (inner dimension contiguous).
int make_tmap_2d_u8(CUtensorMap* map, const void* base, int64_t inner, int64_t outer, int64_t row_stride,
                    int box_inner, int box_outer, int swizzle);
// 3-D uint8 tensor map: dimension 0 contiguous, dimensions 1 and 2 at the
// given byte strides (which may overlap: dimension 2 can step inside 1).
int make_tmap_3d_u8(CUtensorMap* map, const void* base, int64_t d0, int64_t d1, int64_t d2, int64_t stride1,
                    int64_t stride2, int box0, int box1, int box2, int swizzle);
// 2-D 16-bit map (e.g. a bf16 output), rows of row_stride_bytes.
int make_tmap_2d_u16(CUtensorMap* map, const void* base, int64_t inner, int64_t outer, int64_t row_stride_bytes,
                     int box_inner, int box_outer, int swizzle);

// ---- gemm_w4a4.cu: device address of the status word bounded waits write.
int* device_status_ptr();

// ---- quantize.cu
int launch_quantize(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                    float* s_t, int s_t_mode, int scale_layout, void* workspace, cudaStream_t stream);
int launch_prepack_scales(const uint8_t* src, int64_t batch, int64_t rows, int64_t K, uint8_t* dst,
                          cudaStream_t stream);
size_t quantize_workspace_bytes();
// bf16 x [rows][K] -> NVFP4 with MMA-layout scales and s_t = amax / 2688,
// where amax (fp32 bits) was already taken by the kernel that wrote x
// amax_bits = max |x| (fp32 bits) over n bf16 values (n % 8 == 0); zeroes it first
int launch_amax_bf16(const uint16_t* x, int64_t n, unsigned int* amax_bits, cudaStream_t stream);
int launch_quantize_bf16_from_amax(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                                   const unsigned int* amax_bits, float* s_t, cudaStream_t stream);

// ---- gemv.cu
size_t w4a16_workspace_bytes(int64_t M, int64_t N, int64_t K);
size_t argmax_workspace_bytes(int64_t M, int64_t K);
int launch_gemm_w4a16(const uint16_t* X, int64_t M, const nvfp4_tensor_t& W, uint16_t* Y, void* ws,
                      cudaStream_t stream);
int launch_gemm_w4a16_silu_mul(const uint16_t* X, int64_t M, const nvfp4_tensor_t& W, uint16_t* H, void* ws,
                               cudaStream_t stream);
int launch_gather_argmax(const uint16_t* H, int64_t M, const nvfp4_tensor_t& W, const int32_t* idx,
                         int64_t n_idx, int32_t* out_ids, float* out_logit, void* ws, cudaStream_t stream);
int launch_gather_rows(const nvfp4_tensor_t& W, const int32_t* idx, int64_t n_idx, uint8_t* codes_out,
                       uint8_t* scales_out, cudaStream_t stream);
int launch_gemv_argmax(const uint16_t* H, int64_t M, const nvfp4_tensor_t& W, const int32_t* ids,
                       int32_t* out_ids, float* out_logit, void* ws, cudaStream_t stream,
                       const int32_t* draft_ids = nullptr, int n_draft = 0, int32_t* n_accepted = nullptr);

// ---- moe.cu
int launch_moe_route(const float* logits, int64_t T, int E, int topk, int32_t* ids, float* weights,
                     cudaStream_t stream);
size_t grouped_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk);
int launch_grouped_gemm(const uint16_t* X, int64_t T, int topk, const int32_t* ids, const float* w,
                        const nvfp4_tensor_t& W13, const nvfp4_tensor_t& W2, uint16_t* out, void* ws,
                        cudaStream_t stream);
size_t grouped_w4a4_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk);
int launch_grouped_gemm_w4a4(const uint16_t* X, int64_t T, int topk, const int32_t* ids, const float* w,
                             const nvfp4_tensor_t& W13, const nvfp4_tensor_t& W2, uint16_t* out, void* ws,
                             cudaStream_t stream);

// ---- gemm_w4a4.cu
size_t w4a4_workspace_bytes(int64_t M, int64_t N, int64_t K);
int launch_gemm_w4a4(const nvfp4_tensor_t& A, const nvfp4_tensor_t& W, uint16_t* Y, void* ws,
                     cudaStream_t stream);
size_t w4a4_quant_workspace_bytes(int64_t M, int64_t N, int64_t K);
int launch_gemm_w4a4_quant(const nvfp4_tensor_t& A, const nvfp4_tensor_t& W, uint8_t* codes, uint8_t* scales,
                           float* s_t, int s_t_mode, uint16_t* Y, void* ws, cudaStream_t stream);
int read_device_status(int* out, cudaStream_t stream);
int selftest_bounded_wait(int64_t limit_ns, cudaStream_t stream);
int probe_fp4_mma_rate(int n_mma, int n_ctas, cudaStream_t stream);
// Grouped W4A4 expert GEMM over a routing plan's tile table (gate/up with
// SiLU * mul, or down): with `pair`, CTA pairs over tiles of up to W4A4_TILE
// routed rows, else one CTA per tile of up to 128; a_codes / a_scales:
// tile-major routed rows [a_rows][K] (tile t at rows t * tile size);
// h_out / y_out: [out_rows] rows in the plan's order.
constexpr int W4A4_TILE = 256;
int launch_grouped_w4a4(bool gateup, const uint8_t* a_codes, const uint8_t* a_scales, const float* st_a,
                        int64_t a_rows, const nvfp4_tensor_t& W, const int* tile_count, const int* tile_expert,
                        const int* tile_row0, const int* tile_rows, int64_t max_tiles, int inter, int hidden,
                        uint16_t* h_out, unsigned int* amax_bits, uint16_t* y_out, int64_t out_rows, bool pair,
                        cudaStream_t stream);

}  // namespace nvfp4
