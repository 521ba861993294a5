// Host-side launch helpers and the internal interface between the C ABI
// (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

inline int from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

// Number of SMs of the current device (queried once per device).
int sm_count();

// Launch `kernel` with a thread-block cluster of `cluster_x` CTAs along x
// (plain launch when cluster_x == 1).
template <typename Kernel, typename... Args>
int launch_cluster(Kernel kernel, dim3 grid, dim3 block, size_t smem, int cluster_x, cudaStream_t stream,
                   Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (cluster_x > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return from_cuda(cudaLaunchKernelEx(&cfg, kernel, args...));
}

// ---- quantize.cu
int launch_quantize(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                    float* s_t, int s_t_mode, int scale_layout, void* workspace, cudaStream_t stream);
int launch_prepack_scales(const uint8_t* src, int64_t batch, int64_t rows, int64_t K, uint8_t* dst,
                          cudaStream_t stream);
size_t quantize_workspace_bytes();

// ---- gemv.cu
size_t w4a16_workspace_bytes(int64_t M, int64_t K);
size_t argmax_workspace_bytes(int64_t M, int64_t K);
int launch_gemm_w4a16(const uint16_t* X, int64_t M, const nvfp4_tensor_t& W, uint16_t* Y, void* ws,
                      cudaStream_t stream);
int launch_gather_argmax(const uint16_t* H, int64_t M, const nvfp4_tensor_t& W, const int32_t* idx,
                         int64_t n_idx, int32_t* out_ids, float* out_logit, void* ws, cudaStream_t stream);

// ---- moe.cu
int launch_moe_route(const float* logits, int64_t T, int E, int topk, int32_t* ids, float* weights,
                     cudaStream_t stream);
size_t grouped_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk);
int launch_grouped_gemm(const uint16_t* X, int64_t T, int topk, const int32_t* ids, const float* w,
                        const nvfp4_tensor_t& W13, const nvfp4_tensor_t& W2, uint16_t* out, void* ws,
                        cudaStream_t stream);

// ---- gemm_w4a4.cu
size_t w4a4_workspace_bytes(int64_t M, int64_t N, int64_t K);
int launch_gemm_w4a4(const nvfp4_tensor_t& A, const nvfp4_tensor_t& W, uint16_t* Y, void* ws,
                     cudaStream_t stream);
int read_device_status(int* out, cudaStream_t stream);
int selftest_bounded_wait(int64_t limit_ns, cudaStream_t stream);

}  // namespace nvfp4
