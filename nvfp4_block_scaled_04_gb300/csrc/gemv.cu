// Decode W4A16 GEMV / skinny GEMM and the masked draft head's gathered-row
// GEMV with fused argmax. The mainloop lives in gemv_core.cuh; this file
// sizes the launches and carves the workspace.
#include "gemv_core.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

// One CTA per output row of a dense activation matrix X[M][K] (rows beyond
// M, up to the n-tile padding of the chunk, become zeros).
__global__ void __launch_bounds__(GV_THREADS) xprep_dense_kernel(const uint16_t* X, int64_t M, int64_t K,
                                                                  uint4* xfrag, int* pexp) {
  const int64_t out_row = static_cast<int64_t>(blockIdx.y) * GV_MCHUNK + blockIdx.x;
  xprep_row(out_row < M ? X + out_row * K : nullptr, K, out_row, xfrag, pexp);
}

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// CTAs per cluster along K: as many as still fit in one wave of two CTAs
// per SM, so that every CTA is resident at once and HBM bandwidth is shared
// evenly; at most 8 (portable cluster size) and at most one per iteration.
int choose_split(int64_t base_ctas, int64_t n_it) {
  const int64_t cap = 2LL * sm_count();
  int64_t s = cap / (base_ctas > 0 ? base_ctas : 1);
  s = s < 1 ? 1 : s;
  s = s > 8 ? 8 : s;
  s = s > n_it ? n_it : s;
  return static_cast<int>(s);
}

template <int MODE>
int launch_skinny_nt(int nt, const SkinnyParams& p, dim3 grid, cudaStream_t stream) {
  switch (nt) {
    case 1: return launch_cluster(skinny_kernel<1, MODE>, grid, dim3(GV_THREADS), 0, p.split, stream, p);
    case 2: return launch_cluster(skinny_kernel<2, MODE>, grid, dim3(GV_THREADS), 0, p.split, stream, p);
    case 3: return launch_cluster(skinny_kernel<3, MODE>, grid, dim3(GV_THREADS), 0, p.split, stream, p);
    default: return launch_cluster(skinny_kernel<4, MODE>, grid, dim3(GV_THREADS), 0, p.split, stream, p);
  }
}

struct DenseWs {
  int* pexp;
  uint4* xfrag;
  unsigned long long* keys;
  unsigned int* counter;
  size_t bytes;
};

DenseWs carve_dense(void* base, int64_t M, int64_t K, bool argmax) {
  const int64_t chunks = ceil_div(M, GV_MCHUNK);
  DenseWs w{};
  size_t off = 0;
  char* b = static_cast<char*>(base);
  if (argmax) {
    w.keys = reinterpret_cast<unsigned long long*>(b + off);
    off += align_up(GV_MCHUNK * sizeof(unsigned long long));
    w.counter = reinterpret_cast<unsigned int*>(b + off);
    off += kAlign;
  }
  w.pexp = reinterpret_cast<int*>(b + off);
  off += align_up(static_cast<size_t>(chunks) * GV_MCHUNK * sizeof(int));
  w.xfrag = reinterpret_cast<uint4*>(b + off);
  off += align_up(xfrag_bytes(chunks, K));
  w.bytes = off;
  return w;
}

int prep_dense(const uint16_t* X, int64_t M, int64_t K, int nt, const DenseWs& w, cudaStream_t stream) {
  const int64_t chunks = ceil_div(M, GV_MCHUNK);
  dim3 grid(static_cast<unsigned>(8 * nt), static_cast<unsigned>(chunks));
  xprep_dense_kernel<<<grid, GV_THREADS, 0, stream>>>(X, M, K, w.xfrag, w.pexp);
  return from_cuda(cudaGetLastError());
}

}  // namespace

size_t w4a16_workspace_bytes(int64_t M, int64_t K) { return carve_dense(nullptr, M, K, false).bytes; }
size_t argmax_workspace_bytes(int64_t M, int64_t K) { return carve_dense(nullptr, M, K, true).bytes; }

int launch_gemm_w4a16(const uint16_t* X, int64_t M, const nvfp4_tensor_t& W, uint16_t* Y, void* ws,
                      cudaStream_t stream) {
  const int64_t K = W.K, N = W.rows;
  const DenseWs w = carve_dense(ws, M, K, false);
  const int nt = static_cast<int>(ceil_div(M < GV_MCHUNK ? M : GV_MCHUNK, 8));
  int rc = prep_dense(X, M, K, nt, w, stream);
  if (rc != NVFP4_OK) return rc;
  const int64_t n_it = K / GV_KIT;
  const int64_t row_tiles = ceil_div(N, GV_ROWS), chunks = ceil_div(M, GV_MCHUNK);
  SkinnyParams p{};
  p.codes = W.codes;
  p.scales = W.scales;
  p.s_t = W.s_t;
  p.K = K;
  p.n_rows = N;
  p.xfrag = w.xfrag;
  p.pexp = w.pexp;
  p.M = M;
  p.split = choose_split(row_tiles * chunks, n_it);
  p.Y = Y;
  dim3 grid(static_cast<unsigned>(p.split), static_cast<unsigned>(row_tiles), static_cast<unsigned>(chunks));
  return launch_skinny_nt<SK_PLAIN>(nt, p, grid, stream);
}

int launch_gather_argmax(const uint16_t* H, int64_t M, const nvfp4_tensor_t& W, const int32_t* idx,
                         int64_t n_idx, int32_t* out_ids, float* out_logit, void* ws, cudaStream_t stream) {
  const int64_t K = W.K;
  const DenseWs w = carve_dense(ws, M, K, true);
  // keys and the completion counter start at zero on every call
  if (cudaMemsetAsync(w.keys, 0, reinterpret_cast<char*>(w.pexp) - reinterpret_cast<char*>(w.keys), stream) !=
      cudaSuccess)
    return NVFP4_ERR_CUDA;
  const int nt = static_cast<int>(ceil_div(M, 8));
  int rc = prep_dense(H, M, K, nt, w, stream);
  if (rc != NVFP4_OK) return rc;
  const int64_t n_it = K / GV_KIT;
  const int64_t row_tiles = ceil_div(n_idx, GV_ROWS);
  SkinnyParams p{};
  p.codes = W.codes;
  p.scales = W.scales;
  p.s_t = W.s_t;
  p.K = K;
  p.n_rows = n_idx;
  p.idx = idx;
  p.xfrag = w.xfrag;
  p.pexp = w.pexp;
  p.M = M;
  p.split = choose_split(row_tiles, n_it);
  p.keys = w.keys;
  p.counter = w.counter;
  p.out_ids = out_ids;
  p.out_logit = out_logit;
  dim3 grid(static_cast<unsigned>(p.split), static_cast<unsigned>(row_tiles), 1);
  return launch_skinny_nt<SK_ARGMAX>(nt, p, grid, stream);
}

}  // namespace nvfp4
