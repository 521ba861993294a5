// Allocation-free variant of the W4A16 decode linear.
//
// nvfp4_gemm_w4a16 needs a caller-provided workspace for the activations it
// converts to f16. Some callers cannot provide one: a serving engine that
// reserves nearly all device memory for its KV cache at start-up and hands
// kernels no spare buffers, or a host that must not call cudaMalloc /
// cudaFree on its decode path because those calls can synchronise the
// device. For them, nvfp4_gemm_w4a16_noalloc runs the same kernels with the
// scratch held in a fixed array of device memory that this file declares.
//
// Properties a user relies on:
//   - The array below is part of the library image: every GPU that loads the
//     library holds it (8 MiB) until the process exits.
//   - The host never dereferences `g_noalloc_scratch`; in host code that name
//     is only a stand-in. Its device address is looked up once per device
//     with cudaGetSymbolAddress, on the first call made while that device is
//     current, and cached. Make that first call before any stream capture.
//   - Every call shares the one array. Calls whose kernels overlap on the GPU
//     (two streams, or two host threads) race on it and corrupt each other's
//     results; serialise them. Each call rewrites every byte it later reads,
//     so nothing has to start at zero.
//   - Limits: 1 <= M <= 32 tokens and K <= 32768; larger shapes are rejected
//     with NVFP4_ERR_SCRATCH_LIMIT before anything is launched. Within them
//     the scratch a call needs is the split-K partials (one 32 x 128 fp32
//     block per CTA, at most two CTAs per SM: 4.75 MiB on 152 SMs) plus the
//     f16 activation fragments (2 MiB at K = 32768) and a few KiB of shifts
//     and counters, under the 8 MiB of the array; the size is checked on
//     every call, so a GPU with more SMs gets the error rather than an
//     overrun.
//   - The cached address belongs to the device's current module image:
//     after cudaDeviceReset it is stale, so the library must not be used on
//     a device after a reset in the same process.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int64_t kNoallocMaxM = 32;
constexpr int64_t kNoallocMaxK = 32768;
constexpr size_t kNoallocBytes = 8u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return NVFP4_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" int nvfp4_gemm_w4a16_noalloc(const void* X, int64_t M, nvfp4_tensor_t W, void* Y,
                                        nvfp4_stream_t stream) {
  if (!X || !Y || M < 1 || !W.codes || !W.scales || !W.s_t || W.rows < 0 || W.K <= 0 || W.batch != 1 ||
      W.scale_layout != NVFP4_SCALES_ROWMAJOR)
    return NVFP4_ERR_INVALID_ARG;
  if (W.K % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (M > kNoallocMaxM || W.K > kNoallocMaxK || w4a16_workspace_bytes(M, W.rows, W.K) > kNoallocBytes)
    return NVFP4_ERR_SCRATCH_LIMIT;
  if (!aligned16(X) || !aligned16(W.codes) || !aligned16(Y)) return NVFP4_ERR_MISALIGNED;
  if (W.rows == 0) return NVFP4_OK;
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != NVFP4_OK) return rc;
  return launch_gemm_w4a16(static_cast<const uint16_t*>(X), M, W, static_cast<uint16_t*>(Y), scratch,
                           reinterpret_cast<cudaStream_t>(stream));
}
