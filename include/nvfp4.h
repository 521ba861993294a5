/*
 * nvfp4.h - C ABI of libnvfp4.so: the NVFP4 block-scaled linear layer of a
 * 4-bit LLM serving engine, on one NVIDIA GB300 (sm_103a).
 *
 * The format. Values are 4-bit e2m1 codes, and every 16 consecutive elements
 * along K share one 8-bit floating-point block scale (Serving Qwen3.8-27B in
 * 4-bit with a masked speculative decoding head, "What the artifact is"); that
 * scale is E4M3, four exponent and three mantissa bits (What 350+ Experiments
 * Taught Us About Serving Qwen 3.6 35B-A3B, section 3).
 * A tensor T[rows][K] is stored as
 *   codes   uint8 [rows][K/2]   element 2j in the low nibble of byte j,
 *                               element 2j+1 in the high nibble;
 *   scales  uint8 [rows][K/16]  one E4M3 block scale per 16 elements along K
 *                               (row-major; or the MMA layout, see below);
 *   s_t     fp32                 one tensor scale (device memory).
 * and decodes to  x_hat[r][k] = e2m1(code) * e4m3(scale[r][k/16]) * s_t.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless stated otherwise; the caller owns
 *    every buffer. The library allocates nothing.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream); nothing
 *    synchronises the host. Stream order holds for every input: a call
 *    reads nothing before the work enqueued ahead of it has finished. The
 *    decode entry points overlap a call's start with the previous kernel's
 *    drain (programmatic dependent launch) only in ways that keep this true.
 *  - Return value: NVFP4_OK (0) or a negative NVFP4_ERR_*; arguments are
 *    validated on the host before anything is launched, so an error return
 *    means nothing was enqueued (except NVFP4_ERR_CUDA, raised by a failed
 *    launch). The library never aborts and prints nothing.
 *  - bf16 means IEEE-style bfloat16 (uint16 storage), row-major.
 *  - Base pointers of codes, activations and outputs must be 16-byte aligned.
 *  - No CPU fallback exists: every call runs CUDA kernels on the current
 *    device.
 *  - Per device, the library caches device addresses of its own device
 *    variables (the status word, the fixed scratch of the allocation-free
 *    entry point) and kernel attributes on first use. cudaDeviceReset
 *    invalidates them: do not use the library on a device after resetting it
 *    in the same process.
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvfp4_stream_t;   /* == cudaStream_t */

/* ---- status codes ------------------------------------------------------ */
#define NVFP4_OK                     0
#define NVFP4_ERR_INVALID_ARG       -1   /* null pointer, negative size, bad enum */
#define NVFP4_ERR_UNSUPPORTED_SHAPE -2   /* a size is not a multiple of the op's granule */
#define NVFP4_ERR_MISALIGNED        -3   /* a pointer that must be 16-byte aligned is not */
#define NVFP4_ERR_CUDA              -4   /* a CUDA runtime / driver call failed */
#define NVFP4_ERR_WORKSPACE         -5   /* workspace missing or too small */
#define NVFP4_ERR_TIMEOUT           -6   /* a bounded on-device wait gave up (device status word) */
#define NVFP4_ERR_SCRATCH_LIMIT     -7   /* shape exceeds the fixed scratch of nvfp4_gemm_w4a16_noalloc */

/* ---- enums --------------------------------------------------------------- */
#define NVFP4_DTYPE_F32   0
#define NVFP4_DTYPE_BF16  1

#define NVFP4_ST_COMPUTE  0   /* s_t = amax(|x|) / 2688 (1 if all zero), written to *s_t */
#define NVFP4_ST_GIVEN    1   /* s_t read from *s_t (must be finite and > 0) */

/* Scale layouts.
 * ROWMAJOR: scales[r][j] at r*(K/16) + j.
 * MMA: the layout the block-scaled tensor-core MMA consumes. Rows are padded
 *   to a multiple of 128 and the K/16 scale columns to a multiple of 4; the
 *   padded matrix is cut into 128x4 tiles of 512 bytes, tile (rt, ct) at byte
 *   (rt * (Kp/64) + ct) * 512, and inside a tile row r, column c sits at
 *   (r % 32) * 16 + (r / 32) * 4 + c. Padding bytes are zero. */
#define NVFP4_SCALES_ROWMAJOR 0
#define NVFP4_SCALES_MMA      1

/* An NVFP4 tensor (or a stack of `batch` equally shaped ones, e.g. the
 * experts of a MoE layer). Matrix b starts at codes + b*rows*K/2, at
 * scales + b*nvfp4_scales_bytes(rows, K, scale_layout), and its tensor scale
 * is s_t[b] (device memory). */
typedef struct nvfp4_tensor {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* s_t;
  int64_t rows;
  int64_t K;
  int32_t batch;
  int32_t scale_layout;
} nvfp4_tensor_t;

/* Operation ids for nvfp4_workspace_size. */
#define NVFP4_OP_QUANTIZE        0
#define NVFP4_OP_GEMM_W4A16      1
#define NVFP4_OP_GEMM_W4A4       2
#define NVFP4_OP_GROUPED_GEMM    3
#define NVFP4_OP_GATHER_ARGMAX   4
#define NVFP4_OP_GEMM_W4A4_QUANT 5
#define NVFP4_OP_GROUPED_GEMM_W4A4 6

/* ---- entry points ----------------------------------------------------------- */

/* Quantise x[rows][K] (fp32 or bf16) to NVFP4.
 * The per-16 block scale is amax(|block|)/6 rounded to E4M3 (nearest, ties
 * to even, saturating at 448), taken relative to the tensor scale; each
 * element is x / (e4m3(scale) * s_t) rounded to e2m1 (nearest, ties to the
 * even code, saturating at 6; the sign of a negative element is kept even
 * when its magnitude rounds to zero; a zero scale gives zero codes). All
 * decisions are fp32 with IEEE division. The format is the pages' (see the
 * top of this file); the rounding rules are readings of it.
 *   x          device, rows*K elements of x_dtype, 16-byte aligned
 *   codes      device out, rows*K/2 bytes, 16-byte aligned
 *   scales     device out, nvfp4_scales_bytes(rows, K, scale_layout) bytes
 *   s_t        device fp32: written (COMPUTE) or read (GIVEN)
 *   workspace  device, >= nvfp4_workspace_size(NVFP4_OP_QUANTIZE, ...) bytes
 *              (COMPUTE only; may be NULL for GIVEN); contents are scratch.
 * K must be a multiple of 16, and rows * ceil(K / 1024) must stay below 2^30
 * (NVFP4_ERR_UNSUPPORTED_SHAPE otherwise). rows == 0 is a no-op (COMPUTE
 * writes s_t = 1). */
int nvfp4_quantize(const void* x, int x_dtype, int64_t rows, int64_t K,
                   uint8_t* codes, uint8_t* scales, float* s_t, int s_t_mode,
                   int scale_layout, void* workspace, size_t workspace_bytes,
                   nvfp4_stream_t stream);

/* Re-lay row-major block scales into the MMA layout (a one-time weight
 * prepack; activations can be quantised straight into the MMA layout).
 *   src  device, batch*rows*(K/16) bytes, row-major
 *   dst  device, batch*nvfp4_scales_bytes(rows, K, NVFP4_SCALES_MMA) bytes */
int nvfp4_prepack_scales(const uint8_t* src, int64_t batch, int64_t rows, int64_t K,
                         uint8_t* dst, nvfp4_stream_t stream);

/* W4A16 linear (decode): Y[m][n] = bf16( sum_k X[m][k] * W_hat[n][k] ) with
 * fp32 accumulation: 4-bit weights against 16-bit activations, the decode form
 * of the layer (What 350+ Experiments..., section 1; Qwen3.8-27B benchmark,
 * "Serving configuration measured").
 *   X  device bf16 [M][K];  W  NVFP4 [N][K], batch 1, ROWMAJOR scales;
 *   Y  device bf16 [M][N].
 *   workspace  >= nvfp4_workspace_size(NVFP4_OP_GEMM_W4A16, M, N, K) bytes:
 *              the activations converted to f16 (each token times a power of
 *              two that keeps it in f16 range, exact) in MMA fragment order.
 * K must be a multiple of 128. Any M >= 1 (tuned for M <= 32). */
int nvfp4_gemm_w4a16(const void* X, int64_t M, nvfp4_tensor_t W, void* Y,
                     void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Fused gate/up projection of a dense MLP with SiLU * mul in its epilogue:
 * W stacks the gate rows [0, I) and the up rows [I, 2I) (W.rows = 2I), and
 *   H[m][i] = bf16( silu(g) * u ),  g = sum_k X[m][k] W_hat[i][k],
 *                                   u = sum_k X[m][k] W_hat[I + i][k]
 * (g, u fp32-accumulated as in nvfp4_gemm_w4a16; silu(g) = g / (1 + e^-g)).
 * The [M][2I] gate/up output never goes through memory: one round trip of
 * the activations between two linears less, in the 4-bit-weight decoder
 * layers of the pages (52.6% More Tokens..., comparison paragraph; the
 * row order is the one the routed experts use, What 350+ Experiments...,
 * section 1).
 *   X  device bf16 [M][K];  W  NVFP4 [2I][K], batch 1, ROWMAJOR scales;
 *   H  device bf16 [M][I];
 *   workspace  >= nvfp4_workspace_size(NVFP4_OP_GEMM_W4A16, M, 2I, K) bytes.
 * K must be a multiple of 256 and I a multiple of 64. */
int nvfp4_gemm_w4a16_silu_mul(const void* X, int64_t M, nvfp4_tensor_t W, void* H,
                              void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* nvfp4_gemm_w4a16 without a workspace: the same computation and kernels, with
 * the converted activations and split-K partials kept in a fixed 8 MiB array of device
 * memory inside the library instead of caller memory. The pages have no
 * counterpart of this entry point; it serves callers that cannot allocate on
 * their decode path - an engine that reserves nearly all device memory for its
 * KV cache at start-up, or a host that must not call cudaMalloc / cudaFree
 * there because those calls can synchronise the device.
 *   X, M, W, Y as for nvfp4_gemm_w4a16; 1 <= M <= 32, K <= 32768 and the
 *   workspace nvfp4_workspace_size(NVFP4_OP_GEMM_W4A16, M, N, K) would need
 *   at most 8 MiB (true for every such shape on a GPU of up to 152 SMs: the
 *   split-K partials take at most 2 * SMs * 16 KiB, the converted activations
 *   at most 2 MiB); otherwise NVFP4_ERR_SCRATCH_LIMIT before anything is
 *   launched.
 * The first call on each device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress; make it before any
 * stream capture. All calls share the array: calls that overlap on the GPU
 * race and must be serialised by the caller. Nothing in it needs zeroing. */
int nvfp4_gemm_w4a16_noalloc(const void* X, int64_t M, nvfp4_tensor_t W, void* Y,
                             nvfp4_stream_t stream);

/* W4A4 linear (prefill): Y[m][n] = bf16( s_tA * s_tW * sum_k a[m][k] * w[n][k] )
 * where a, w are the e2m1*e4m3 products, multiplied and accumulated (fp32) by
 * the block-scaled FP4 tensor cores: both operands 4-bit, run natively on
 * Blackwell (52.6% More Tokens, 1.53x Less GPU Time: Production Inference
 * with Minima and Rafay, comparison paragraph).
 *   A  NVFP4 [M][K] (typically from nvfp4_quantize, COMPUTE);
 *   W  NVFP4 [N][K]; both batch 1. MMA-layout scales are used in place;
 *      ROWMAJOR scales are re-laid into the workspace first.
 *   Y  device bf16 [M][N].
 *   workspace >= nvfp4_workspace_size(NVFP4_OP_GEMM_W4A4, M, N, K) when an
 *      operand has ROWMAJOR scales; unused (may be NULL) otherwise.
 * K must be a multiple of 64 and N a multiple of 8; M >= 1 arbitrary. */
int nvfp4_gemm_w4a4(nvfp4_tensor_t A, nvfp4_tensor_t W, void* Y,
                    void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* W4A4 linear whose output goes on as NVFP4, the input of the next W4A4
 * layer: W4A4 end to end, with no bf16 activation between the two linears
 * making a round trip through memory in the fused case (52.6% More
 * Tokens..., comparison paragraph). The output is the quantisation (the
 * rules of nvfp4_quantize, MMA-layout scales) of the bf16 output
 * Y = bf16(s_tA * s_tW * sum_k a * w) that nvfp4_gemm_w4a4 would write:
 *   NVFP4_ST_GIVEN    *s_t is the output's tensor scale (a static,
 *                     calibrated one): one fused kernel, whose epilogue
 *                     quantises each row's 16-column blocks; Y is not written
 *                     and may be NULL.
 *   NVFP4_ST_COMPUTE  s_t = amax(|Y|) / 2688 (1 if Y is all zero), written to
 *                     *s_t: a tensor-wide amax is needed before any block can
 *                     be encoded, so the GEMM writes Y (bf16, caller buffer
 *                     [M][N]) and folds its amax on the fly, and a second
 *                     kernel encodes Y without another amax pass.
 *   A, W       as for nvfp4_gemm_w4a4; N (W.rows) a multiple of 64
 *   codes      device out [M][N/2];  scales device out, nvfp4_scales_bytes(M, N,
 *              NVFP4_SCALES_MMA) bytes (padding bytes written as zero)
 *   workspace  >= nvfp4_workspace_size(NVFP4_OP_GEMM_W4A4_QUANT, M, N, K). */
int nvfp4_gemm_w4a4_quant(nvfp4_tensor_t A, nvfp4_tensor_t W, uint8_t* codes, uint8_t* scales, float* s_t,
                          int s_t_mode, void* Y, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Top-k routing of a MoE layer: p = softmax(logits[t]) (fp32), the k experts
 * with the largest p (ties to the lower expert id), weights = those p (not
 * renormalised). ids int32 [T][topk], weights fp32 [T][topk], in descending
 * p order. E <= 1024, topk <= 32. */
int nvfp4_moe_route(const float* logits, int64_t T, int E, int topk,
                    int32_t* ids, float* weights, nvfp4_stream_t stream);

/* Routed-expert MoE layer, W4A16 (What 350+ Experiments..., sections 1 and 7:
 * NVFP4 mixture-of-experts operations):
 *   for each token t and slot j with e = topk_ids[t][j]:
 *     [g; u] = X[t] @ W13_e^T      (W13_e rows [0, I) gate, [I, 2I) up)
 *     h      = bf16( silu(g) * u )
 *     y      = bf16( h @ W2_e^T )  (fp32 accumulation)
 *     out[t] += topk_w[t][j] * y
 *   out = bf16(sum over j, fp32, in slot order).
 *   X        device bf16 [T][H];  topk_ids int32 [T][topk]: a slot whose id
 *            lies outside [0, E) is dropped (it adds nothing to out[t]) and
 *            sets NVFP4_ERR_INVALID_ARG in the device status word
 *            (nvfp4_read_device_status);
 *   topk_w   fp32 [T][topk];
 *   W13      NVFP4, batch E, rows 2I, K H, ROWMAJOR;
 *   W2       NVFP4, batch E, rows H,  K I, ROWMAJOR;
 *   out      device bf16 [T][H];
 *   workspace >= nvfp4_workspace_size(NVFP4_OP_GROUPED_GEMM, T, H, I, E, topk).
 * H and I must be multiples of 128; E <= 4096. Layers whose experts get at
 * least 32 routed rows on average (T * topk >= 32 E), with H and I multiples
 * of 256, run the expert GEMMs on the tensor cores; others on the streaming
 * kernel. Both compute the products exactly and sum in fp32 (the summation
 * order differs between them). Repeated calls with the same inputs give
 * identical outputs. */
int nvfp4_grouped_gemm(const void* X, int64_t T, int topk, const int32_t* topk_ids,
                       const float* topk_w, nvfp4_tensor_t W13, nvfp4_tensor_t W2,
                       void* out, void* workspace, size_t workspace_bytes,
                       nvfp4_stream_t stream);

/* The routed-expert MoE layer of nvfp4_grouped_gemm with 4-bit activations
 * as well (W4A4 on the block-scaled FP4 tensor cores; What 350+
 * Experiments..., sections 1 and 7, where the final configuration serves the
 * experts with an NVFP4 MoE kernel). Readings where the pages are silent:
 *   - the layer input X is quantised once per call with its own dynamic
 *     tensor scale (amax / 2688, the quantiser's rules); each routed row is
 *     its token's quantised row;
 *   - [g; u] = x_hat @ W13_e^T, h = bf16(silu(g) * u) as in the W4A16 layer;
 *   - the h rows of all routed (token, slot) pairs are quantised together,
 *     one dynamic tensor scale per call, before the down projection;
 *   - out[t] = bf16(sum_j w[t][j] * y[t][j]), fp32, slots in order
 *     (deterministic).
 *   X, topk_ids, topk_w, out as for nvfp4_grouped_gemm (an expert id outside
 *   [0, E) is dropped and reported the same way);
 *   W13, W2    NVFP4 stacks as for nvfp4_grouped_gemm, with MMA-layout scales
 *              (nvfp4_prepack_scales, batch = E);
 *   workspace  >= nvfp4_workspace_size(NVFP4_OP_GROUPED_GEMM_W4A4, T, H, I, E, topk).
 * H must be a multiple of 256 and I of 128; E <= 4096. */
int nvfp4_grouped_gemm_w4a4(const void* X, int64_t T, int topk, const int32_t* topk_ids, const float* topk_w,
                            nvfp4_tensor_t W13, nvfp4_tensor_t W2, void* out, void* workspace,
                            size_t workspace_bytes, nvfp4_stream_t stream);

/* Masked draft LM head: gathered-row GEMV with a fused argmax. The draft
 * proposes only ids from a fixed subset of the vocabulary, so the head reads
 * only those rows ("The masked head trick", Serving Qwen3.8-27B...):
 *   logit[m][j] = sum_k H[m][k] * W_hat[idx[j]][k]   (fp32 accumulation)
 *   out_ids[m]  = idx[argmax_j logit[m][j]], ties to the lowest vocabulary id
 *   out_logit[m] = that maximum logit (fp32), if out_logit != NULL.
 *   H      device bf16 [M][K];  W  NVFP4 [V][K], batch 1, ROWMAJOR;
 *   idx    device int32 [n_idx]; NULL = every row (n_idx = V). An entry
 *          outside [0, V) is skipped: that row is never read and never
 *          reported; if no entry is valid, out_ids[m] = -1 and out_logit[m]
 *          is a NaN.
 *   workspace >= nvfp4_workspace_size(NVFP4_OP_GATHER_ARGMAX, M, n_idx, K, 0, 0).
 * K must be a multiple of 128; 1 <= M <= 32; n_idx >= 1. */
int nvfp4_gather_gemv_argmax(const void* H, int64_t M, nvfp4_tensor_t W,
                             const int32_t* idx, int64_t n_idx, int32_t* out_ids,
                             float* out_logit, void* workspace, size_t workspace_bytes,
                             nvfp4_stream_t stream);

/* Compact copy of selected rows of an NVFP4 matrix: row j of the output is
 * row idx[j] of W (its packed codes and its row-major block scales; the
 * tensor scale is W's and stays with the caller). A one-time prepack for a
 * fixed row subset such as the draft head's mask ("The masked head trick",
 * Serving Qwen3.8-27B...), so that every draft step then streams the subset as
 * one dense matrix.
 *   W           NVFP4 [V][K], batch 1, ROWMAJOR scales; K a multiple of 32
 *   idx         device int32 [n_idx]; an entry outside [0, V) yields a zero row
 *               and sets NVFP4_ERR_INVALID_ARG in the device status word
 *               (nvfp4_read_device_status)
 *   codes_out   device, n_idx * K/2 bytes, 16-byte aligned
 *   scales_out  device, n_idx * K/16 bytes */
int nvfp4_gather_rows(nvfp4_tensor_t W, const int32_t* idx, int64_t n_idx, uint8_t* codes_out,
                      uint8_t* scales_out, nvfp4_stream_t stream);

/* GEMV with a fused argmax over every row of W, reporting ids through a map:
 *   logit[m][j]  = sum_k H[m][k] * W_hat[j][k]   (fp32 accumulation)
 *   out_ids[m]   = ids[argmax_j logit[m][j]] (j when ids == NULL); among equal
 *                  logits the lowest reported id wins
 *   out_logit[m] = that maximum logit, if out_logit != NULL.
 * With W the nvfp4_gather_rows copy of a head's masked rows and ids the mask,
 * this is the masked draft head of nvfp4_gather_gemv_argmax on a compact
 * matrix (same result, same bytes streamed per step).
 *   H   device bf16 [M][K], 1 <= M <= 32;  W NVFP4, batch 1, ROWMAJOR,
 *       K a multiple of 256;  ids device int32 [W.rows] or NULL
 *   workspace >= nvfp4_workspace_size(NVFP4_OP_GATHER_ARGMAX, M, W.rows, K, 0, 0). */
int nvfp4_gemv_argmax(const void* H, int64_t M, nvfp4_tensor_t W, const int32_t* ids, int32_t* out_ids,
                      float* out_logit, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Speculative verify head: the full-vocabulary GEMV + argmax of
 * nvfp4_gemv_argmax over every row of the LM head W, with a batched greedy
 * acceptance of the drafts fused into its last step. The draft proposes from
 * the masked head, verification reads the whole vocabulary (Serving
 * Qwen3.8-27B in 4-bit..., "The masked head trick"); the verify change of
 * the Qwen3.8-27B benchmark ("Sustained mixed load") is this step.
 *   H           device bf16 [batch * (n_draft + 1)][K]: row b * (n_draft + 1)
 *               + i is sequence b at position i (the last accepted token, then
 *               its n_draft drafts); batch * (n_draft + 1) <= 32
 *   W           NVFP4 [V][K], batch 1, ROWMAJOR, K a multiple of 256
 *   draft_ids   device int32 [batch][n_draft]: the drafted ids; draft i of a
 *               sequence is checked against the argmax at its position i
 *   out_tokens  device int32 [batch][n_draft + 1]: the argmax (lowest id among
 *               equal logits) at every position
 *   n_accepted  device int32 [batch]: the number of leading drafts equal to
 *               out_tokens at the same position; the step emits
 *               out_tokens[b][0 .. n_accepted[b]] (the accepted drafts and one
 *               token from the target)
 *   workspace  >= nvfp4_workspace_size(NVFP4_OP_GATHER_ARGMAX, batch * (n_draft + 1), V, K, 0, 0). */
int nvfp4_verify_accept(const void* H, int64_t batch, int n_draft, nvfp4_tensor_t W, const int32_t* draft_ids,
                        int32_t* out_tokens, int32_t* n_accepted, void* workspace, size_t workspace_bytes,
                        nvfp4_stream_t stream);

/* ---- helpers --------------------------------------------------------------- */

/* Bytes of one matrix's block scales in the given layout. */
size_t nvfp4_scales_bytes(int64_t rows, int64_t K, int scale_layout);

/* Workspace bytes an operation needs (0 if none). Arguments by op:
 *   QUANTIZE:      (rows, -, K, -, -)
 *   GEMM_W4A16:    (M, N, K, -, -)
 *   GEMM_W4A4:     (M, N, K, -, -)   (worst case: both operands ROWMAJOR)
 *   GROUPED_GEMM:  (T, H, I, E, topk)
 *   GATHER_ARGMAX: (M, n_idx, K, -, -)
 *   GEMM_W4A4_QUANT: (M, N, K, -, -)
 *   GROUPED_GEMM_W4A4: (T, H, I, E, topk) */
size_t nvfp4_workspace_size(int op, int64_t a, int64_t b, int64_t c, int64_t e, int64_t topk);

/* Human-readable name of a status code (static storage). */
const char* nvfp4_status_string(int status);

/* Reads and clears the device status word (synchronises `stream`). Bounded
 * on-device waits that give up set NVFP4_ERR_TIMEOUT; nvfp4_gather_rows and
 * nvfp4_grouped_gemm set NVFP4_ERR_INVALID_ARG for an index outside the
 * matrix / an expert id outside [0, E). *out = NVFP4_OK or
 * the last status set. */
int nvfp4_read_device_status(int* out, nvfp4_stream_t stream);

/* Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier nothing will ever arrive on, giving up after `limit_ns`
 * nanoseconds, and records the outcome in the device status word. Used by the
 * tests to show that a wait that runs out returns an error instead of hanging. */
int nvfp4_selftest_bounded_wait(int64_t limit_ns, nvfp4_stream_t stream);

/* Measurement helper (no counterpart on the pages): the issue-rate ceiling of
 * the block-scaled FP4 tensor cores on this GPU. Launches n_ctas CTAs (0 = one
 * per SM), each issuing n_mma tcgen05.mma.kind::mxf4nvf4 instructions of
 * 128 x 256 x 64 (2 * 128 * 256 * 64 flop each, the instruction of the W4A4
 * kernels) into one tensor-memory accumulator from zero-filled shared memory,
 * with no global memory traffic. The caller times the launch (e.g. with CUDA
 * events on `stream`); flop / time is the rate the tensor pipe sustains.
 * 1 <= n_mma <= 2^20, n_ctas >= 0. */
int nvfp4_probe_fp4_mma_rate(int n_mma, int n_ctas, nvfp4_stream_t stream);

/* Library version (major * 10000 + minor * 100 + patch). */
int nvfp4_version(void);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_H_ */
