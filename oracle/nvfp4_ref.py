"""CPU oracle for the NVFP4 block-scaled linear layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs use it. It shares no code with the CUDA path.

What it computes, and the passages it follows
---------------------------------------------
* The format: 4-bit e2m1 values, one 8-bit float scale per 16 consecutive
  elements (Serving Qwen3.8-27B in 4-bit with a masked speculative decoding
  head, "What the artifact is"). That scale is E4M3, an 8-bit float with 4
  exponent and 3 mantissa bits (What 350+ Experiments Taught Us About Serving
  Qwen 3.6 35B-A3B, section 3 "KV cache and memory capacity").
  A second, FP32 per-tensor scale multiplies every decoded value.
* W4A16: 4-bit weights against 16-bit activations (What 350+ Experiments...,
  section 1 "Checkpoint packages and quantisation"; Qwen3.8-27B benchmark,
  "Serving configuration measured").
* W4A4: both operands NVFP4, run natively on Blackwell (52.6% More Tokens,
  1.53x Less GPU Time: Production Inference with Minima and Rafay, comparison
  paragraph).
* Routed-expert MoE layer (What 350+ Experiments..., section 1 and section 7,
  where the final configuration runs the expert GEMMs on an NVFP4 MoE kernel).
* Masked draft LM head: the draft proposes only ids from a fixed 32,768-id
  subset of the 248,320-row head; verification stays full-vocabulary, so the
  mask cannot alter what the model emits (Serving Qwen3.8-27B..., "The masked
  head trick").

Readings where the pages are silent:
  R1 tensor scale  s_t = amax(|x|) / 2688 in fp32 (2688 = 6 * 448); s_t = 1
     when the tensor is all zeros.
  R2 block scale   d = fp32(s_t * 6); sb = fp32(amax_block / d);
     scale = E4M3(sb), round to nearest, ties to even, saturating at 448.
  R3 element code  den = fp32(e4m3(scale) * s_t); q = fp32(x / den);
     code = e2m1(q), nearest, ties to the even code, |q| > 6 saturates to 6.
     A negative x (including -0.0) keeps its sign bit even when its magnitude
     rounds to zero. A block whose scale is 0x00 gets all-zero codes.
  R4 packing       byte j of a row holds element 2j in its low nibble and
     element 2j+1 in its high nibble; scales row-major [rows][K/16].
  R5 GEMMs         plain fp64 sums of the decoded operands. W4A4 decodes the
     quantised activations (the quantiser is pinned bit-exactly on its own).
  R6 argmax        ties go to the lowest vocabulary id; the result is the
     vocabulary id, not the position in the mask.
  R7 MoE           softmax in fp64, top-k by probability with ties to the lower
     expert id, weights = the chosen probabilities (not renormalised);
     W13 rows [0, I) are the gate, [I, 2I) the up projection;
     h = bf16(silu(g) * u); out = sum_j w_j * (h_j @ W2_e^T).
     Each expert matrix carries its own tensor scale.
  R11 verify       speculative verification is greedy: sequence b's rows
     are its n_draft + 1 positions; the target token at position i is the
     full-vocabulary argmax there (R6); the drafts are accepted up to the
     first one that differs from the target token at its position, and the
     step emits the accepted drafts plus the target token after them.
  R12 NVFP4 out    a W4A4 layer whose output feeds the next W4A4 layer hands
     on the quantisation (R1-R3) of its bf16 output; with a static tensor
     scale that scale is given, with a dynamic one it is amax/2688 of the
     whole bf16 output.
  R10 W4A4 MoE     (the routed experts with 4-bit activations as well): the
     layer input is quantised once per call with its own dynamic tensor scale
     and each routed row is its token's quantised row; h as in R7; the h rows
     of all routed (token, slot) pairs are quantised together, one dynamic
     tensor scale per call, before the down projection.

The quantiser takes its decisions in fp32 (numpy float32 arithmetic is IEEE
round-to-nearest-even with no fused multiply-add), the precision the GPU
kernels use for the same decisions. Everything downstream is fp64.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32

# ---------------------------------------------------------------------------
# Codecs, from the bit definitions of the two minifloat formats.
# ---------------------------------------------------------------------------

def e2m1_value(code):
    """Value of a 4-bit e2m1 code: bit 3 sign, bits 2..1 exponent (bias 1),
    bit 0 mantissa. Exponent 0 is subnormal: m * 0.5."""
    c = np.asarray(code, dtype=np.int64) & 0xF
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m / 2.0, e - 1))
    return np.where(s == 1, -mag, mag).astype(np.float64)


def e4m3_value(code):
    """Value of an FP8 E4M3 ("fn" variant) code: bit 7 sign, bits 6..3
    exponent (bias 7), bits 2..0 mantissa. Exponent 0 is subnormal
    (m/8 * 2^-6). 0x7F and 0xFF are NaN; there are no infinities."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag).astype(np.float64)


# Non-negative finite codes in increasing value order (codes are monotonic in
# value for a fixed sign, so the table is simply the code range).
_E2M1_POS_CODES = np.arange(8, dtype=np.int64)
_E2M1_POS_VALUES = e2m1_value(_E2M1_POS_CODES)
_E4M3_POS_CODES = np.arange(0x7F, dtype=np.int64)          # 0x00 .. 0x7E
_E4M3_POS_VALUES = e4m3_value(_E4M3_POS_CODES)


def _nearest_even(mag, values, codes):
    """Nearest representable value to each non-negative `mag` (float64 array
    of values exactly representable from fp32); a tie between two neighbours
    goes to the even code; anything at or above the largest value saturates."""
    mag = np.asarray(mag, dtype=np.float64)
    n = len(values)
    hi = np.clip(np.searchsorted(values, mag, side="left"), 0, n - 1)
    lo = np.clip(hi - 1, 0, n - 1)
    d_lo = mag - values[lo]
    d_hi = values[hi] - mag
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    return np.where(take_hi, codes[hi], codes[lo])


def e4m3_encode(x):
    """fp32 (>= 0) -> E4M3 code, round to nearest, ties to even, saturating
    values above 448 (infinity included) to 448 (0x7E). Scales are never
    negative."""
    x = np.asarray(x, dtype=np.float32)
    if np.any(np.isnan(x)) or np.any(x < 0):
        raise ValueError("block scales are non-negative and not NaN")
    return _nearest_even(x.astype(np.float64), _E4M3_POS_VALUES, _E4M3_POS_CODES).astype(np.uint8)


def e2m1_encode(q):
    """fp32 -> e2m1 code: magnitude by nearest-with-ties-to-even over
    {0, .5, 1, 1.5, 2, 3, 4, 6}, saturating at 6; the sign bit copies the sign
    bit of q (so -0.0 and small negatives give 0x8)."""
    q = np.asarray(q, dtype=np.float32)
    if np.any(np.isnan(q)):
        raise ValueError("e2m1_encode: NaN input")
    mag = _nearest_even(np.abs(q).astype(np.float64), _E2M1_POS_VALUES, _E2M1_POS_CODES)
    return (mag | (np.signbit(q).astype(np.int64) << 3)).astype(np.uint8)


# ---------------------------------------------------------------------------
# Quantise / decode a [rows][K] tensor.
# ---------------------------------------------------------------------------

class QTensor:
    """An NVFP4 tensor in the exported layout: codes uint8 [rows][K/2]
    (element 2j low nibble, 2j+1 high nibble), scales uint8 [rows][K/16]
    (E4M3), s_t float32."""

    def __init__(self, codes, scales, s_t):
        self.codes = np.ascontiguousarray(codes, dtype=np.uint8)
        self.scales = np.ascontiguousarray(scales, dtype=np.uint8)
        self.s_t = F32(s_t)

    @property
    def shape(self):
        return self.codes.shape[0], self.codes.shape[1] * 2

    def rows(self, idx):
        return QTensor(self.codes[idx], self.scales[idx], self.s_t)


def tensor_scale(x):
    """R1: s_t = fp32(amax / 2688), or 1 for an all-zero tensor."""
    x = np.asarray(x, dtype=np.float32)
    amax = F32(np.max(np.abs(x))) if x.size else F32(0)
    if amax == 0:
        return F32(1.0)
    return F32(amax / F32(2688.0))


def pack_codes(codes):
    """R4: [rows][K] 4-bit codes -> [rows][K/2] bytes."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def quantize(x, s_t=None):
    """Quantise a [rows][K] tensor (fp32 values; bf16 inputs are exact in fp32)
    to NVFP4, following R1-R4 step by step. `s_t` given -> used as is
    (static scale); None -> computed from the tensor (R1)."""
    x = np.asarray(x, dtype=np.float32)
    if x.ndim != 2 or x.shape[1] % 16 != 0:
        raise ValueError("quantize wants [rows][K] with K a multiple of 16")
    R, K = x.shape
    st = tensor_scale(x) if s_t is None else F32(s_t)
    blocks = x.reshape(R, K // 16, 16)
    amax_b = np.max(np.abs(blocks), axis=2) if R else np.zeros((0, K // 16), np.float32)
    d = F32(st * F32(6.0))
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        sb = (amax_b / d).astype(np.float32)
    scale = e4m3_encode(sb)
    den = (e4m3_value(scale).astype(np.float32) * st).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        q = (blocks / den[:, :, None]).astype(np.float32)
    zero_blk = scale == 0
    q = np.where(zero_blk[:, :, None], F32(0.0), q)
    codes = e2m1_encode(q.reshape(R, K))
    codes = np.where(np.repeat(zero_blk, 16, axis=1), np.uint8(0), codes).astype(np.uint8)
    return QTensor(pack_codes(codes), scale, st)


def decode(qt: QTensor):
    """x_hat = e2m1(code) * e4m3(scale) * s_t, in fp64 (exact)."""
    codes = unpack_codes(qt.codes)
    R, K = codes.shape
    v = e2m1_value(codes).reshape(R, K // 16, 16)
    s = e4m3_value(qt.scales)[:, :, None]
    return (v * s * np.float64(qt.s_t)).reshape(R, K)


# ---------------------------------------------------------------------------
# The linear layers.
# ---------------------------------------------------------------------------

def gemm_w4a16(x, w: QTensor):
    """Y[m][n] = sum_k x[m][k] * w_hat[n][k], fp64. x holds the bf16 inputs."""
    return np.asarray(x, dtype=np.float64) @ decode(w).T


def gemm_w4a4(a: QTensor, w: QTensor):
    """Y = A_hat @ W_hat^T in fp64 on two quantised operands (R5)."""
    return decode(a) @ decode(w).T


def gemm_w4a4_nvfp4(a: QTensor, w: QTensor, s_t=None):
    """R12: the W4A4 output as NVFP4 for the next W4A4 layer: quantise(bf16(
    A_hat @ W_hat^T)), tensor scale given or (None) dynamic."""
    y = bf16_round(gemm_w4a4(a, w)).astype(np.float32)   # bf16 values are exact in fp32
    return quantize(y, s_t=s_t)


def bf16_round(v):
    """Round fp64 values to the nearest bf16 (8 significant bits), ties to
    even, in one step (no intermediate fp32 rounding). Normal range only."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                       # v = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


def rel_fro(y, y_ref):
    """||y - y_ref||_F / ||y_ref||_F."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    den = np.linalg.norm(y_ref)
    return float(np.linalg.norm(y - y_ref) / den) if den > 0 else float(np.linalg.norm(y))


# ---------------------------------------------------------------------------
# Masked draft head: gathered-row GEMV + argmax.
# ---------------------------------------------------------------------------

def gather_logits(h, w: QTensor, idx=None):
    """Logits over the candidate rows (idx, or every row), fp64 [M][n]."""
    rows = np.arange(w.codes.shape[0]) if idx is None else np.asarray(idx, dtype=np.int64)
    return np.asarray(h, dtype=np.float64) @ decode(w.rows(rows)).T, rows


def argmax_lowest_id(logits, rows):
    """R6: per row of `logits`, the vocabulary id of the largest logit; among
    equal maxima the lowest id. Returns (ids int64 [M], max logit fp64 [M])."""
    logits = np.asarray(logits, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    mx = logits.max(axis=1)
    ids = np.array([rows[logits[i] == mx[i]].min() for i in range(logits.shape[0])], dtype=np.int64)
    return ids, mx


def gather_gemv_argmax(h, w: QTensor, idx=None):
    logits, rows = gather_logits(h, w, idx)
    ids, mx = argmax_lowest_id(logits, rows)
    return ids, mx, logits


def top2_margin(logits):
    """(l1 - l2) / RMS(l) per row: how far the winner stands clear."""
    logits = np.asarray(logits, dtype=np.float64)
    s = np.sort(logits, axis=1)
    rms = np.sqrt(np.mean(logits ** 2, axis=1))
    return (s[:, -1] - s[:, -2]) / rms


def accept_greedy(target_ids, draft_ids):
    """R11: per sequence, the number of leading drafts equal to the target
    token at the same position. target_ids [B][D+1], draft_ids [B][D]."""
    target_ids = np.asarray(target_ids, dtype=np.int64)
    draft_ids = np.asarray(draft_ids, dtype=np.int64)
    B, D = draft_ids.shape
    n = np.zeros(B, dtype=np.int64)
    for b in range(B):
        while n[b] < D and draft_ids[b, n[b]] == target_ids[b, n[b]]:
            n[b] += 1
    return n


def verify_accept(h, w: QTensor, draft_ids):
    """Speculative verify step (R11): full-vocabulary logits of the
    B * (D + 1) hidden rows, the target token per position (R6), and the
    accepted draft count per sequence. Returns (target ids [B][D+1], accepted
    [B], logits [B*(D+1)][V])."""
    draft_ids = np.asarray(draft_ids, dtype=np.int64)
    B, D = draft_ids.shape
    ids, _, logits = gather_gemv_argmax(h, w, None)
    target = ids.reshape(B, D + 1)
    return target, accept_greedy(target, draft_ids), logits


# ---------------------------------------------------------------------------
# Routed-expert MoE layer.
# ---------------------------------------------------------------------------

def moe_route(logits, topk):
    """R7 routing: fp64 softmax over experts, the top-k experts by probability
    (ties -> lower expert id), weights = their probabilities."""
    z = np.asarray(logits, dtype=np.float64)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    T, E = p.shape
    ids = np.empty((T, topk), dtype=np.int64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-p[t, e], e))
        ids[t] = order[:topk]
    return ids, np.take_along_axis(p, ids, axis=1)


def silu(g):
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):   # exp(-g) = inf for g << 0 gives the right limit, 0
        return g / (1.0 + np.exp(-g))


def moe_forward(x, ids, weights, w13: list, w2: list):
    """R7: out[t] = sum_j w[t,j] * (bf16(silu(g) * u) @ W2_e^T) with
    [g; u] = x[t] @ W13_e^T, e = ids[t, j]. w13 / w2 are per-expert QTensors."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(ids)
    weights = np.asarray(weights, dtype=np.float64)
    T, H = x.shape
    out = np.zeros((T, w2[0].shape[0]), dtype=np.float64)
    for e in range(len(w13)):
        tok, slot = np.nonzero(ids == e)
        if tok.size == 0:
            continue
        gu = x[tok] @ decode(w13[e]).T
        inter = gu.shape[1] // 2
        h = bf16_round(silu(gu[:, :inter]) * gu[:, inter:])
        y = h @ decode(w2[e]).T
        np.add.at(out, tok, weights[tok, slot][:, None] * y)
    return out


def moe_forward_w4a4(x, ids, weights, w13: list, w2: list):
    """R10: the R7 layer with NVFP4 activations into both expert projections
    (What 350+ Experiments..., section 7: the NVFP4 mixture-of-experts
    kernels). x_hat = decode(quantise(x)) with one dynamic tensor scale for the
    call; [g; u] = x_hat[t] @ W13_e^T; h = bf16(silu(g) * u) for every routed
    (t, j); h_hat = decode(quantise(all routed h rows)), one dynamic tensor
    scale for the call; out[t] = sum_j w[t,j] * (h_hat[t,j] @ W2_e^T).
    Decoded products summed in fp64 (R5)."""
    x = np.asarray(x, dtype=np.float32)
    ids = np.asarray(ids)
    weights = np.asarray(weights, dtype=np.float64)
    T = x.shape[0]
    xd = decode(quantize(x))
    tok, slot = np.nonzero((ids >= 0) & (ids < len(w13)))
    exp = ids[tok, slot]
    inter = w13[0].shape[0] // 2
    h = np.zeros((tok.size, inter), dtype=np.float64)
    for e in np.unique(exp):
        r = np.nonzero(exp == e)[0]
        gu = xd[tok[r]] @ decode(w13[e]).T
        h[r] = bf16_round(silu(gu[:, :inter]) * gu[:, inter:])
    hd = decode(quantize(h.astype(np.float32))) if tok.size else h   # bf16 values are exact in fp32
    out = np.zeros((T, w2[0].shape[0]), dtype=np.float64)
    for e in np.unique(exp):
        r = np.nonzero(exp == e)[0]
        y = hd[r] @ decode(w2[e]).T
        np.add.at(out, tok[r], weights[tok[r], slot[r]][:, None] * y)
    return out
