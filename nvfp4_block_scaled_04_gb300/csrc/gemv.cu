// Decode W4A16 GEMV / skinny GEMM and the masked draft head's gathered-row
// GEMV with fused argmax. The mainloop lives in gemv_core.cuh; this file
// sizes the launches and carves the workspace.
#include "gemv_core.cuh"
#include "gemv_tma.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

// One CTA per output row of a dense activation matrix X[M][K] (rows beyond
// M, up to the n-tile padding of the chunk, become zeros).
// CTA (0, 0) also zeroes the split-K arrival counters (or the argmax keys and
// completion counter) of the kernel that follows.
// 1024 threads per row: up to K = 32768 the row is read once, into registers.
// Launched as a programmatic dependent of whatever kernel precedes it on the
// stream, so it is resident and waiting while that kernel drains. Once that
// kernel has finished (its writes visible) it lets its own GEMV launch, which
// starts streaming its weights (and reading the index of gathered rows)
// while this kernel converts the activations: everything enqueued before the
// call is complete before the GEMV reads any of its inputs.
constexpr int XPREP_THREADS = 1024;
__global__ void __launch_bounds__(XPREP_THREADS) xprep_dense_kernel(const uint16_t* X, int64_t M, int64_t K,
                                                                     uint4* xfrag, int* pexp,
                                                                     unsigned int* counters, int n_counters) {
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0u;
  const int64_t out_row = static_cast<int64_t>(blockIdx.y) * GV_MCHUNK + blockIdx.x;
  const uint16_t* src = out_row < M ? X + out_row * K : nullptr;
  const int64_t n8 = K / 8;
  if (n8 <= XPREP_THREADS) xprep_row_regs<1>(src, K, out_row, xfrag, pexp);
  else if (n8 <= 2 * XPREP_THREADS) xprep_row_regs<2>(src, K, out_row, xfrag, pexp);
  else if (n8 <= 4 * XPREP_THREADS) xprep_row_regs<4>(src, K, out_row, xfrag, pexp);
  else xprep_row(src, K, out_row, xfrag, pexp);
}

// Row j of the compact copy = row idx[j] of W (codes and row-major scales),
// one warp per row, 16-byte copies. An index outside [0, rows) gives a zero
// row and NVFP4_ERR_INVALID_ARG in the device status word.
__global__ void gather_rows_kernel(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t K,
                                   const int32_t* idx, int64_t n_idx, uint8_t* codes_out, uint8_t* scales_out,
                                   int* status) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (j >= n_idx) return;
  const int64_t v = idx[j];
  const bool ok = v >= 0 && v < rows;
  if (!ok && lane == 0) atomicExch(status, NVFP4_ERR_INVALID_ARG);
  const int64_t kb = K / 2, ks = K / 16;
  const uint4* src = reinterpret_cast<const uint4*>(codes + (ok ? v : 0) * kb);
  uint4* dst = reinterpret_cast<uint4*>(codes_out + j * kb);
  for (int64_t q = lane; q < kb / 16; q += 32) dst[q] = ok ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
  for (int64_t q = lane; q < ks; q += 32) scales_out[j * ks + q] = ok ? scales[v * ks + q] : 0;
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

// One warp layout for every token count: two m-tiles per consumer warp (each
// activation fragment read from shared memory feeds two MMAs) and the stage's
// two K-iterations on two warps. A token's output is then summed in the same
// order whatever the batch size, so its bits do not depend on which other
// tokens share the call.
template <int NT>
int launch_tma_plain_nt(const TmaSkinnyParams& p, const CUtensorMap& mc, const CUtensorMap& ms, dim3 grid,
                        cudaStream_t stream) {
  constexpr int MT = 2;
  constexpr int KW = 2;
  auto k = skinny_tma_kernel<NT, SK_PLAIN, MT, KW>;
  int rc = ensure_smem(k, GtCfg<NT>::SMEM);
  if (rc != NVFP4_OK) return rc;
  return launch_ex(k, grid, dim3(GtWarps<MT, KW>::THREADS), GtCfg<NT>::SMEM, 1, true, stream, mc, ms, p);
}

// GEMV with argmax on the TMA-fed kernel (split 1). With an index the codes
// and scales come in by tile::gather4 of one-row-high boxes (GATHER), over
// the whole weight by 2-D boxes of 128 rows. The plain GEMV's warp layout at
// every token count: a row's logit is summed in the order the unsplit GEMV
// sums that output, so its bits do not depend on the batch, and rounded to
// bf16 it is the GEMV's output for that row.
template <int NT, bool GATHER>
int launch_tma_argmax_nt(const TmaSkinnyParams& p, const CUtensorMap& mc, const CUtensorMap& ms, dim3 grid,
                         cudaStream_t stream) {
  constexpr int MT = 2;
  constexpr int KW = 2;
  using C = GtCfg<NT, GATHER ? GT_SCALES_GATHERED : GT_SCALES>;
  auto k = skinny_tma_kernel<NT, SK_ARGMAX, MT, KW, GATHER>;
  int rc = ensure_smem(k, C::SMEM);
  if (rc != NVFP4_OK) return rc;
  return launch_ex(k, grid, dim3(GtWarps<MT, KW>::THREADS), C::SMEM, 1, true, stream, mc, ms, p);
}

// Split-K of the TMA-fed GEMV: as many K-slices per 128-row tile as still fit
// in one wave of two CTAs per SM (at most 8, at least one stage each). It is
// chosen from the 128-row tiles of ONE token chunk, so it depends on (N, K)
// alone: a token's partial sums and their reduction order are the same at
// every M (calls with more than 32 tokens run one such wave per chunk).
int tma_split(int64_t row_tiles, int64_t n_stages) { return choose_split(row_tiles, n_stages); }

struct DenseWs {
  int* pexp;
  uint4* xfrag;
  unsigned long long* keys;
  unsigned int* counter;
  unsigned int* tile_counters;
  int n_tile_counters;
  float* partials;
  size_t bytes;
};

// Workspace: [argmax keys + counter] [per-token shifts] [split-K counters]
// [split-K partials] [activation fragments].
DenseWs carve_dense(void* base, int64_t M, int64_t N, int64_t K, bool argmax) {
  const int64_t chunks = ceil_div(M, GV_MCHUNK);
  DenseWs w{};
  size_t off = 0;
  char* b = static_cast<char*>(base);
  if (argmax) {
    // keys and completion counter, contiguous: the prep kernel zeroes them as 32-bit words
    w.keys = reinterpret_cast<unsigned long long*>(b + off);
    off += align_up(GV_MCHUNK * sizeof(unsigned long long));
    w.counter = reinterpret_cast<unsigned int*>(b + off);
    off += kAlign;
    w.tile_counters = reinterpret_cast<unsigned int*>(w.keys);
    w.n_tile_counters = static_cast<int>(off / sizeof(unsigned int));
  }
  w.pexp = reinterpret_cast<int*>(b + off);
  off += align_up(static_cast<size_t>(chunks) * GV_MCHUNK * sizeof(int));
  if (!argmax && K % 256 == 0) {
    // only a split tile needs counters and partials; then per token chunk
    // row tiles * split <= 2 * SMs
    const int64_t tiles = chunks * ceil_div(N, GV_ROWS);
    const int S = tma_split(ceil_div(N, GV_ROWS), K / 256);
    if (S > 1) {
      w.n_tile_counters = static_cast<int>(tiles);
      w.tile_counters = reinterpret_cast<unsigned int*>(b + off);
      off += align_up(static_cast<size_t>(tiles) * sizeof(unsigned int));
      w.partials = reinterpret_cast<float*>(b + off);
      off += align_up(static_cast<size_t>(tiles) * S * GV_MCHUNK * GV_ROWS * sizeof(float));
    }
  }
  w.xfrag = reinterpret_cast<uint4*>(b + off);
  off += align_up(xfrag_bytes(chunks, K));
  w.bytes = off;
  return w;
}

int prep_dense(const uint16_t* X, int64_t M, int64_t K, int nt, const DenseWs& w, cudaStream_t stream) {
  const int64_t chunks = ceil_div(M, GV_MCHUNK);
  dim3 grid(static_cast<unsigned>(8 * nt), static_cast<unsigned>(chunks));
  return launch_ex(xprep_dense_kernel, grid, dim3(XPREP_THREADS), 0, 1, true, stream, X, M, K, w.xfrag, w.pexp,
                   w.tile_counters, w.n_tile_counters);
}

}  // namespace

size_t w4a16_workspace_bytes(int64_t M, int64_t N, int64_t K) { return carve_dense(nullptr, M, N, K, false).bytes; }
size_t argmax_workspace_bytes(int64_t M, int64_t K) { return carve_dense(nullptr, M, 0, K, true).bytes; }

int launch_gemm_w4a16(const uint16_t* X, int64_t M, const nvfp4_tensor_t& W, uint16_t* Y, void* ws,
                      cudaStream_t stream) {
  const int64_t K = W.K, N = W.rows;
  const DenseWs w = carve_dense(ws, M, N, K, false);
  const int nt = static_cast<int>(ceil_div(M < GV_MCHUNK ? M : GV_MCHUNK, 8));
  int rc = prep_dense(X, M, K, nt, w, stream);
  if (rc != NVFP4_OK) return rc;
  const int64_t n_it = K / GV_KIT;
  const int64_t row_tiles = ceil_div(N, GV_ROWS), chunks = ceil_div(M, GV_MCHUNK);
  if (K % 256 == 0) {
    // TMA-fed kernel: codes and scales stream through a shared-memory ring
    CUtensorMap mc, ms;
    rc = make_tmap_2d_u8(&mc, W.codes, K / 2, N, K / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != NVFP4_OK) return rc;
    rc = make_tmap_2d_u8(&ms, W.scales, K / 16, N, K / 16, 16, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != NVFP4_OK) return rc;
    TmaSkinnyParams q{};
    q.s_t = W.s_t;
    q.K = K;
    q.n_rows = N;
    q.xfrag = w.xfrag;
    q.pexp = w.pexp;
    q.M = M;
    q.split = tma_split(row_tiles, n_it / 2);
    q.Y = Y;
    q.status = device_status_ptr();
    q.partials = w.partials;
    q.counters = w.tile_counters;
    dim3 grid(static_cast<unsigned>(q.split), static_cast<unsigned>(row_tiles), static_cast<unsigned>(chunks));
    switch (nt) {
      case 1: return launch_tma_plain_nt<1>(q, mc, ms, grid, stream);
      case 2: return launch_tma_plain_nt<2>(q, mc, ms, grid, stream);
      case 3: return launch_tma_plain_nt<3>(q, mc, ms, grid, stream);
      default: return launch_tma_plain_nt<4>(q, mc, ms, grid, stream);
    }
  }
  SkinnyParams p{};
  p.codes = W.codes;
  p.scales = W.scales;
  p.s_t = W.s_t;
  p.K = K;
  p.n_rows = N;
  p.xfrag = w.xfrag;
  p.pexp = w.pexp;
  p.M = M;
  p.split = choose_split(row_tiles, n_it);   // from (N, K) alone, as for the TMA-fed kernel
  p.Y = Y;
  dim3 grid(static_cast<unsigned>(p.split), static_cast<unsigned>(row_tiles), static_cast<unsigned>(chunks));
  return launch_skinny_nt<SK_PLAIN>(nt, p, grid, stream);
}

// Dense gate/up projection with SiLU * mul fused: W [2I][K], gate rows
// [0, I), up rows [I, 2I); tiles of 64 gate rows and the matching 64 up
// rows, so each CTA holds both halves of its outputs; h = bf16(silu(g) * u).
// The split along K, the warp layout and the reduction order are those of
// the plain GEMV (the split is chosen from the 2I / 128 tiles of (N, K)).
int launch_gemm_w4a16_silu_mul(const uint16_t* X, int64_t M, const nvfp4_tensor_t& W, uint16_t* H, void* ws,
                               cudaStream_t stream) {
  const int64_t K = W.K, N = W.rows, I = N / 2;
  const DenseWs w = carve_dense(ws, M, N, K, false);
  const int nt = static_cast<int>(ceil_div(M < GV_MCHUNK ? M : GV_MCHUNK, 8));
  int rc = prep_dense(X, M, K, nt, w, stream);
  if (rc != NVFP4_OK) return rc;
  const int64_t row_tiles = I / 64, chunks = ceil_div(M, GV_MCHUNK);
  CUtensorMap mc, ms;
  rc = make_tmap_2d_u8(&mc, W.codes, K / 2, N, K / 2, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != NVFP4_OK) return rc;
  rc = make_tmap_2d_u8(&ms, W.scales, K / 16, N, K / 16, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != NVFP4_OK) return rc;
  TmaSkinnyParams q{};
  q.s_t = W.s_t;
  q.K = K;
  q.n_rows = N;
  q.xfrag = w.xfrag;
  q.pexp = w.pexp;
  q.M = M;
  q.split = tma_split(row_tiles, K / 256);
  q.inter = I;
  q.h_out = H;
  q.status = device_status_ptr();
  q.partials = w.partials;
  q.counters = w.tile_counters;
  dim3 grid(static_cast<unsigned>(q.split), static_cast<unsigned>(row_tiles), static_cast<unsigned>(chunks));
  auto launch = [&](auto kernel, int smem) {
    int r = ensure_smem(kernel, smem);
    if (r != NVFP4_OK) return r;
    return launch_ex(kernel, grid, dim3(GtWarps<2, 2>::THREADS), smem, 1, true, stream, mc, ms, q);
  };
  switch (nt) {
    case 1: return launch(skinny_tma_kernel<1, SK_GATEUP_DENSE, 2, 2>, GtCfg<1>::SMEM);
    case 2: return launch(skinny_tma_kernel<2, SK_GATEUP_DENSE, 2, 2>, GtCfg<2>::SMEM);
    case 3: return launch(skinny_tma_kernel<3, SK_GATEUP_DENSE, 2, 2>, GtCfg<3>::SMEM);
    default: return launch(skinny_tma_kernel<4, SK_GATEUP_DENSE, 2, 2>, GtCfg<4>::SMEM);
  }
}

int launch_gather_rows(const nvfp4_tensor_t& W, const int32_t* idx, int64_t n_idx, uint8_t* codes_out,
                       uint8_t* scales_out, cudaStream_t stream) {
  constexpr int kWarps = 8;
  const int64_t blocks = ceil_div(n_idx, kWarps);
  gather_rows_kernel<<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(
      W.codes, W.scales, W.rows, W.K, idx, n_idx, codes_out, scales_out, device_status_ptr());
  return from_cuda(cudaGetLastError());
}

// GEMV + argmax over every row of W (consecutive rows through 2-D TMA boxes);
// row j is reported as ids[j] (j when ids is null). With n_accepted the call
// is a speculative verify head (see TmaSkinnyParams).
int launch_gemv_argmax(const uint16_t* H, int64_t M, const nvfp4_tensor_t& W, const int32_t* ids,
                       int32_t* out_ids, float* out_logit, void* ws, cudaStream_t stream,
                       const int32_t* draft_ids, int n_draft, int32_t* n_accepted) {
  const int64_t K = W.K;
  const DenseWs w = carve_dense(ws, M, 0, K, true);   // keys and counter zeroed by the prep kernel
  const int nt = static_cast<int>(ceil_div(M, 8));
  int rc = prep_dense(H, M, K, nt, w, stream);
  if (rc != NVFP4_OK) return rc;
  CUtensorMap mc, ms;
  rc = make_tmap_2d_u8(&mc, W.codes, K / 2, W.rows, K / 2, 128, GV_ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != NVFP4_OK) return rc;
  rc = make_tmap_2d_u8(&ms, W.scales, K / 16, W.rows, K / 16, 16, GV_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != NVFP4_OK) return rc;
  TmaSkinnyParams q{};
  q.s_t = W.s_t;
  q.K = K;
  q.n_rows = W.rows;
  q.xfrag = w.xfrag;
  q.pexp = w.pexp;
  q.M = M;
  q.split = 1;
  q.status = device_status_ptr();
  q.idx = ids;
  q.keys = w.keys;
  q.counter = w.counter;
  q.out_ids = out_ids;
  q.out_logit = out_logit;
  q.draft_ids = draft_ids;
  q.n_draft = n_draft;
  q.n_accepted = n_accepted;
  const dim3 grid(1, static_cast<unsigned>(ceil_div(W.rows, GV_ROWS)), 1);
  switch (nt) {
    case 1: return launch_tma_argmax_nt<1, false>(q, mc, ms, grid, stream);
    case 2: return launch_tma_argmax_nt<2, false>(q, mc, ms, grid, stream);
    case 3: return launch_tma_argmax_nt<3, false>(q, mc, ms, grid, stream);
    default: return launch_tma_argmax_nt<4, false>(q, mc, ms, grid, stream);
  }
}

int launch_gather_argmax(const uint16_t* H, int64_t M, const nvfp4_tensor_t& W, const int32_t* idx,
                         int64_t n_idx, int32_t* out_ids, float* out_logit, void* ws, cudaStream_t stream) {
  const int64_t K = W.K;
  const DenseWs w = carve_dense(ws, M, 0, K, true);
  // keys and the completion counter start at zero on every call: the prep kernel zeroes them
  const int nt = static_cast<int>(ceil_div(M, 8));
  int rc = prep_dense(H, M, K, nt, w, stream);
  if (rc != NVFP4_OK) return rc;
  const int64_t n_it = K / GV_KIT;
  const int64_t row_tiles = ceil_div(n_idx, GV_ROWS);
  const RsLayout rs = rs_layout(K);
  if (idx && nt == 1 && K % 256 == 0 && rs.smem <= 227 * 1024) {
    // masked rows, one n-tile: stream whole candidate rows
    TmaSkinnyParams q{};
    q.s_t = W.s_t;
    q.K = K;
    q.n_rows = n_idx;
    q.xfrag = w.xfrag;
    q.pexp = w.pexp;
    q.M = M;
    q.split = 1;
    q.status = device_status_ptr();
    q.idx = idx;
    q.w_rows = W.rows;
    q.keys = w.keys;
    q.counter = w.counter;
    q.out_ids = out_ids;
    q.out_logit = out_logit;
    q.codes = W.codes;
    q.scales = W.scales;
    rc = ensure_smem(gather_rows_argmax_kernel, rs.smem);
    if (rc != NVFP4_OK) return rc;
    const int64_t groups = ceil_div(n_idx, RS_ROWS);
    const int64_t grid = groups < sm_count() ? groups : sm_count();
    return launch_ex(gather_rows_argmax_kernel, dim3(static_cast<unsigned>(grid)), dim3(RS_THREADS), rs.smem, 1, true,
                     stream, q, rs);
  }
  if (K % 256 == 0) {
    CUtensorMap mc, ms;
    const int box_rows = idx ? 1 : GV_ROWS;
    rc = make_tmap_2d_u8(&mc, W.codes, K / 2, W.rows, K / 2, 128, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != NVFP4_OK) return rc;
    rc = make_tmap_2d_u8(&ms, W.scales, K / 16, W.rows, K / 16, 16, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != NVFP4_OK) return rc;
    TmaSkinnyParams q{};
    q.s_t = W.s_t;
    q.K = K;
    q.n_rows = n_idx;
    q.xfrag = w.xfrag;
    q.pexp = w.pexp;
    q.M = M;
    q.split = 1;
    q.status = device_status_ptr();
    q.idx = idx;
    q.w_rows = W.rows;
    q.keys = w.keys;
    q.counter = w.counter;
    q.out_ids = out_ids;
    q.out_logit = out_logit;
    const dim3 grid(1, static_cast<unsigned>(row_tiles), 1);
    if (idx) {
      switch (nt) {
        case 1: return launch_tma_argmax_nt<1, true>(q, mc, ms, grid, stream);
        case 2: return launch_tma_argmax_nt<2, true>(q, mc, ms, grid, stream);
        case 3: return launch_tma_argmax_nt<3, true>(q, mc, ms, grid, stream);
        default: return launch_tma_argmax_nt<4, true>(q, mc, ms, grid, stream);
      }
    }
    switch (nt) {
      case 1: return launch_tma_argmax_nt<1, false>(q, mc, ms, grid, stream);
      case 2: return launch_tma_argmax_nt<2, false>(q, mc, ms, grid, stream);
      case 3: return launch_tma_argmax_nt<3, false>(q, mc, ms, grid, stream);
      default: return launch_tma_argmax_nt<4, false>(q, mc, ms, grid, stream);
    }
  }
  SkinnyParams p{};
  p.codes = W.codes;
  p.scales = W.scales;
  p.s_t = W.s_t;
  p.K = K;
  p.n_rows = n_idx;
  p.idx = idx;
  p.w_rows = W.rows;
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
