// The C ABI of libnvfp4.so (declared in include/nvfp4.h): argument
// validation on the host, then dispatch to the kernel files. Nothing here
// computes on the CPU; an invalid call returns an error before any launch.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace nvfp4 {

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

int ensure_smem_impl(const void* func, int bytes) {
  // per (kernel, device): the largest dynamic shared-memory size set so far
  // (a kernel whose size depends on the shape may need more on a later call)
  constexpr int kMaxFuncs = 256, kMaxDevs = 64;
  static std::mutex mu;
  static const void* funcs[kMaxFuncs];
  static int set_bytes[kMaxFuncs][kMaxDevs];
  static int n = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevs) return NVFP4_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(mu);
  int i = 0;
  while (i < n && funcs[i] != func) ++i;
  if (i < n && set_bytes[i][dev] >= bytes) return NVFP4_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  if (i == n) {
    if (n == kMaxFuncs) return NVFP4_OK;
    funcs[n] = func;
    for (int d = 0; d < kMaxDevs; ++d) set_bytes[n][d] = 0;
    ++n;
  }
  set_bytes[i][dev] = bytes;
  return NVFP4_OK;
}

namespace {

bool tensor_ok(const nvfp4_tensor_t& t) {
  return t.codes && t.scales && t.s_t && t.rows >= 0 && t.K > 0 && t.batch >= 1 &&
         (t.scale_layout == NVFP4_SCALES_ROWMAJOR || t.scale_layout == NVFP4_SCALES_MMA);
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

int nvfp4_version(void) { return 100; }

const char* nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case NVFP4_ERR_MISALIGNED: return "misaligned pointer (16-byte alignment required)";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_ERR_TIMEOUT: return "bounded on-device wait timed out";
    case NVFP4_ERR_SCRATCH_LIMIT: return "shape exceeds the fixed scratch of the allocation-free entry point";
    default: return "unknown status";
  }
}

size_t nvfp4_scales_bytes(int64_t rows, int64_t K, int scale_layout) {
  if (rows < 0 || K < 0) return 0;
  if (scale_layout == NVFP4_SCALES_MMA) return static_cast<size_t>(mma_scale_rows(rows) * mma_scale_cols(K));
  return static_cast<size_t>(rows * (K / 16));
}

size_t nvfp4_workspace_size(int op, int64_t a, int64_t b, int64_t c, int64_t e, int64_t topk) {
  if (a < 0 || b < 0 || c < 0 || e < 0 || topk < 0) return 0;
  switch (op) {
    case NVFP4_OP_QUANTIZE: return quantize_workspace_bytes();
    case NVFP4_OP_GEMM_W4A16: return a > 0 && c > 0 ? w4a16_workspace_bytes(a, b, c) : 0;
    case NVFP4_OP_GEMM_W4A4: return w4a4_workspace_bytes(a, b, c);
    case NVFP4_OP_GEMM_W4A4_QUANT: return w4a4_quant_workspace_bytes(a, b, c);
    case NVFP4_OP_GROUPED_GEMM_W4A4: return grouped_w4a4_workspace_bytes(a, b, c, e, topk);
    case NVFP4_OP_GROUPED_GEMM: return grouped_workspace_bytes(a, b, c, e, topk);
    case NVFP4_OP_GATHER_ARGMAX: return a > 0 && c > 0 ? argmax_workspace_bytes(a, c) : 0;
    default: return 0;
  }
}

int nvfp4_quantize(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                   float* s_t, int s_t_mode, int scale_layout, void* workspace, size_t workspace_bytes,
                   nvfp4_stream_t stream) {
  if (!s_t || rows < 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
  if (x_dtype != NVFP4_DTYPE_F32 && x_dtype != NVFP4_DTYPE_BF16) return NVFP4_ERR_INVALID_ARG;
  if (s_t_mode != NVFP4_ST_COMPUTE && s_t_mode != NVFP4_ST_GIVEN) return NVFP4_ERR_INVALID_ARG;
  if (scale_layout != NVFP4_SCALES_ROWMAJOR && scale_layout != NVFP4_SCALES_MMA) return NVFP4_ERR_INVALID_ARG;
  if (K % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (rows > 0 && (!x || !codes || !scales)) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && (!aligned16(x) || !aligned16(codes))) return NVFP4_ERR_MISALIGNED;
  if (s_t_mode == NVFP4_ST_COMPUTE && (!workspace || workspace_bytes < quantize_workspace_bytes()))
    return NVFP4_ERR_WORKSPACE;
  return launch_quantize(x, x_dtype, rows, K, codes, scales, s_t, s_t_mode, scale_layout, workspace,
                         reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_prepack_scales(const uint8_t* src, int64_t batch, int64_t rows, int64_t K, uint8_t* dst,
                         nvfp4_stream_t stream) {
  if (!src || !dst || batch < 1 || rows < 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
  if (K % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return launch_prepack_scales(src, batch, rows, K, dst, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_gemm_w4a16(const void* X, int64_t M, nvfp4_tensor_t W, void* Y, void* workspace,
                     size_t workspace_bytes, nvfp4_stream_t stream) {
  if (!X || !Y || M < 0 || !tensor_ok(W) || W.batch != 1) return NVFP4_ERR_INVALID_ARG;
  if (W.scale_layout != NVFP4_SCALES_ROWMAJOR) return NVFP4_ERR_INVALID_ARG;
  if (W.K % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(X) || !aligned16(W.codes) || !aligned16(Y)) return NVFP4_ERR_MISALIGNED;
  if (M == 0 || W.rows == 0) return NVFP4_OK;
  if (!workspace || workspace_bytes < w4a16_workspace_bytes(M, W.rows, W.K)) return NVFP4_ERR_WORKSPACE;
  return launch_gemm_w4a16(static_cast<const uint16_t*>(X), M, W, static_cast<uint16_t*>(Y), workspace,
                           reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_gemm_w4a16_silu_mul(const void* X, int64_t M, nvfp4_tensor_t W, void* H, void* workspace,
                              size_t workspace_bytes, nvfp4_stream_t stream) {
  if (!X || !H || M < 0 || !tensor_ok(W) || W.batch != 1) return NVFP4_ERR_INVALID_ARG;
  if (W.scale_layout != NVFP4_SCALES_ROWMAJOR) return NVFP4_ERR_INVALID_ARG;
  if (W.K % 256 != 0 || W.rows % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(X) || !aligned16(W.codes) || !aligned16(H)) return NVFP4_ERR_MISALIGNED;
  if (M == 0 || W.rows == 0) return NVFP4_OK;
  if (!workspace || workspace_bytes < w4a16_workspace_bytes(M, W.rows, W.K)) return NVFP4_ERR_WORKSPACE;
  return launch_gemm_w4a16_silu_mul(static_cast<const uint16_t*>(X), M, W, static_cast<uint16_t*>(H), workspace,
                                    reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_gemm_w4a4(nvfp4_tensor_t A, nvfp4_tensor_t W, void* Y, void* workspace, size_t workspace_bytes,
                    nvfp4_stream_t stream) {
  if (!Y || !tensor_ok(A) || !tensor_ok(W) || A.batch != 1 || W.batch != 1) return NVFP4_ERR_INVALID_ARG;
  if (A.K != W.K) return NVFP4_ERR_INVALID_ARG;
  if (A.K % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A.codes) || !aligned16(W.codes) || !aligned16(Y) || !aligned16(A.scales) ||
      !aligned16(W.scales))
    return NVFP4_ERR_MISALIGNED;
  if (A.rows == 0 || W.rows == 0) return NVFP4_OK;
  if (W.rows % 8 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;  // bf16 output rows in 16-byte units
  const bool relayout = A.scale_layout == NVFP4_SCALES_ROWMAJOR || W.scale_layout == NVFP4_SCALES_ROWMAJOR;
  if (relayout && (!workspace || workspace_bytes < w4a4_workspace_bytes(A.rows, W.rows, A.K)))
    return NVFP4_ERR_WORKSPACE;
  return launch_gemm_w4a4(A, W, static_cast<uint16_t*>(Y), workspace, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_gemm_w4a4_quant(nvfp4_tensor_t A, nvfp4_tensor_t W, uint8_t* codes, uint8_t* scales, float* s_t,
                          int s_t_mode, void* Y, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  if (!codes || !scales || !s_t || !tensor_ok(A) || !tensor_ok(W) || A.batch != 1 || W.batch != 1)
    return NVFP4_ERR_INVALID_ARG;
  if (s_t_mode != NVFP4_ST_COMPUTE && s_t_mode != NVFP4_ST_GIVEN) return NVFP4_ERR_INVALID_ARG;
  if (s_t_mode == NVFP4_ST_COMPUTE && !Y) return NVFP4_ERR_INVALID_ARG;
  if (A.K != W.K) return NVFP4_ERR_INVALID_ARG;
  if (A.K % 64 != 0 || W.rows % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A.codes) || !aligned16(W.codes) || !aligned16(A.scales) || !aligned16(W.scales) ||
      !aligned16(codes) || !aligned16(scales) || (Y && !aligned16(Y)))
    return NVFP4_ERR_MISALIGNED;
  if (A.rows == 0 || W.rows == 0) return NVFP4_OK;
  if (!workspace || workspace_bytes < w4a4_quant_workspace_bytes(A.rows, W.rows, A.K)) return NVFP4_ERR_WORKSPACE;
  return launch_gemm_w4a4_quant(A, W, codes, scales, s_t, s_t_mode, static_cast<uint16_t*>(Y), workspace,
                                reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_moe_route(const float* logits, int64_t T, int E, int topk, int32_t* ids, float* weights,
                    nvfp4_stream_t stream) {
  if (!logits || !ids || !weights || T < 0 || E < 1 || E > 1024 || topk < 1 || topk > 32 || topk > E)
    return NVFP4_ERR_INVALID_ARG;
  return launch_moe_route(logits, T, E, topk, ids, weights, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_grouped_gemm(const void* X, int64_t T, int topk, const int32_t* topk_ids, const float* topk_w,
                       nvfp4_tensor_t W13, nvfp4_tensor_t W2, void* out, void* workspace, size_t workspace_bytes,
                       nvfp4_stream_t stream) {
  if (!X || !topk_ids || !topk_w || !out || T < 0 || topk < 1 || !tensor_ok(W13) || !tensor_ok(W2))
    return NVFP4_ERR_INVALID_ARG;
  if (W13.scale_layout != NVFP4_SCALES_ROWMAJOR || W2.scale_layout != NVFP4_SCALES_ROWMAJOR)
    return NVFP4_ERR_INVALID_ARG;
  const int64_t E = W13.batch, I = W13.rows / 2, H = W13.K;
  if (W13.rows % 2 != 0 || W2.batch != E || W2.rows != H || W2.K != I || topk > E) return NVFP4_ERR_INVALID_ARG;
  if (H % 128 != 0 || I % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(X) || !aligned16(out) || !aligned16(W13.codes) || !aligned16(W2.codes))
    return NVFP4_ERR_MISALIGNED;
  if (T == 0) return NVFP4_OK;
  if (!workspace || workspace_bytes < grouped_workspace_bytes(T, H, I, E, topk)) return NVFP4_ERR_WORKSPACE;
  return launch_grouped_gemm(static_cast<const uint16_t*>(X), T, topk, topk_ids, topk_w, W13, W2,
                             static_cast<uint16_t*>(out), workspace, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_grouped_gemm_w4a4(const void* X, int64_t T, int topk, const int32_t* topk_ids, const float* topk_w,
                            nvfp4_tensor_t W13, nvfp4_tensor_t W2, void* out, void* workspace, size_t workspace_bytes,
                            nvfp4_stream_t stream) {
  if (!X || !topk_ids || !topk_w || !out || T < 0 || topk < 1 || !tensor_ok(W13) || !tensor_ok(W2))
    return NVFP4_ERR_INVALID_ARG;
  if (W13.scale_layout != NVFP4_SCALES_MMA || W2.scale_layout != NVFP4_SCALES_MMA) return NVFP4_ERR_INVALID_ARG;
  const int64_t E = W13.batch, I = W13.rows / 2, H = W13.K;
  if (W13.rows % 2 != 0 || W2.batch != E || W2.rows != H || W2.K != I || topk > E) return NVFP4_ERR_INVALID_ARG;
  if (H % 256 != 0 || I % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(X) || !aligned16(out) || !aligned16(W13.codes) || !aligned16(W2.codes) || !aligned16(W13.scales) ||
      !aligned16(W2.scales))
    return NVFP4_ERR_MISALIGNED;
  if (T == 0) return NVFP4_OK;
  if (!workspace || workspace_bytes < grouped_w4a4_workspace_bytes(T, H, I, E, topk)) return NVFP4_ERR_WORKSPACE;
  return launch_grouped_gemm_w4a4(static_cast<const uint16_t*>(X), T, topk, topk_ids, topk_w, W13, W2,
                                  static_cast<uint16_t*>(out), workspace, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_gather_gemv_argmax(const void* H, int64_t M, nvfp4_tensor_t W, const int32_t* idx, int64_t n_idx,
                             int32_t* out_ids, float* out_logit, void* workspace, size_t workspace_bytes,
                             nvfp4_stream_t stream) {
  if (!H || !out_ids || M < 1 || M > 32 || !tensor_ok(W) || W.batch != 1) return NVFP4_ERR_INVALID_ARG;
  if (W.scale_layout != NVFP4_SCALES_ROWMAJOR) return NVFP4_ERR_INVALID_ARG;
  if (idx == nullptr) n_idx = W.rows;
  if (n_idx < 1) return NVFP4_ERR_INVALID_ARG;
  if (W.K % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(H) || !aligned16(W.codes)) return NVFP4_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < argmax_workspace_bytes(M, W.K)) return NVFP4_ERR_WORKSPACE;
  return launch_gather_argmax(static_cast<const uint16_t*>(H), M, W, idx, n_idx, out_ids, out_logit, workspace,
                              reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_gather_rows(nvfp4_tensor_t W, const int32_t* idx, int64_t n_idx, uint8_t* codes_out,
                      uint8_t* scales_out, nvfp4_stream_t stream) {
  if (!idx || !codes_out || !scales_out || n_idx < 0 || !tensor_ok(W) || W.batch != 1) return NVFP4_ERR_INVALID_ARG;
  if (W.scale_layout != NVFP4_SCALES_ROWMAJOR) return NVFP4_ERR_INVALID_ARG;
  if (W.K % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;   // whole 16-byte pieces of codes per row
  if (!aligned16(W.codes) || !aligned16(codes_out)) return NVFP4_ERR_MISALIGNED;
  if (n_idx == 0) return NVFP4_OK;
  return launch_gather_rows(W, idx, n_idx, codes_out, scales_out, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_gemv_argmax(const void* H, int64_t M, nvfp4_tensor_t W, const int32_t* ids, int32_t* out_ids,
                      float* out_logit, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  if (!H || !out_ids || M < 1 || M > 32 || !tensor_ok(W) || W.batch != 1 || W.rows < 1) return NVFP4_ERR_INVALID_ARG;
  if (W.scale_layout != NVFP4_SCALES_ROWMAJOR) return NVFP4_ERR_INVALID_ARG;
  if (W.K % 256 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(H) || !aligned16(W.codes) || !aligned16(W.scales)) return NVFP4_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < argmax_workspace_bytes(M, W.K)) return NVFP4_ERR_WORKSPACE;
  return launch_gemv_argmax(static_cast<const uint16_t*>(H), M, W, ids, out_ids, out_logit, workspace,
                            reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_verify_accept(const void* H, int64_t batch, int n_draft, nvfp4_tensor_t W, const int32_t* draft_ids,
                        int32_t* out_tokens, int32_t* n_accepted, void* workspace, size_t workspace_bytes,
                        nvfp4_stream_t stream) {
  if (!H || !out_tokens || !n_accepted || batch < 1 || n_draft < 0 || !tensor_ok(W) || W.batch != 1 || W.rows < 1)
    return NVFP4_ERR_INVALID_ARG;
  if (n_draft > 0 && !draft_ids) return NVFP4_ERR_INVALID_ARG;
  const int64_t M = batch * (n_draft + 1);
  if (M > 32) return NVFP4_ERR_INVALID_ARG;
  if (W.scale_layout != NVFP4_SCALES_ROWMAJOR) return NVFP4_ERR_INVALID_ARG;
  if (W.K % 256 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(H) || !aligned16(W.codes) || !aligned16(W.scales)) return NVFP4_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < argmax_workspace_bytes(M, W.K)) return NVFP4_ERR_WORKSPACE;
  return launch_gemv_argmax(static_cast<const uint16_t*>(H), M, W, nullptr, out_tokens, nullptr, workspace,
                            reinterpret_cast<cudaStream_t>(stream), draft_ids, n_draft, n_accepted);
}

int nvfp4_read_device_status(int* out, nvfp4_stream_t stream) {
  if (!out) return NVFP4_ERR_INVALID_ARG;
  return read_device_status(out, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_probe_fp4_mma_rate(int n_mma, int n_ctas, nvfp4_stream_t stream) {
  // at most 2^20 instructions (tens of milliseconds), far inside the kernel's 2 s bounded wait
  if (n_mma < 1 || n_mma > (1 << 20) || n_ctas < 0) return NVFP4_ERR_INVALID_ARG;
  return probe_fp4_mma_rate(n_mma, n_ctas, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_selftest_bounded_wait(int64_t limit_ns, nvfp4_stream_t stream) {
  if (limit_ns < 1) return NVFP4_ERR_INVALID_ARG;
  return selftest_bounded_wait(limit_ns, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
