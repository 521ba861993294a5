"""Python binding of libnvfp4.so, the NVFP4 block-scaled linear layer for GB300.

Argument marshalling only: every step runs in the library's CUDA kernels
(declared in include/nvfp4.h). PyTorch provides device memory and the current
stream. There is no CPU fallback: if the library is not built, or no CUDA
device is present, every call raises.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from pathlib import Path

import torch

LIB_PATH = Path(__file__).resolve().parent / "libnvfp4.so"

OK = 0
ERR_INVALID_ARG, ERR_TIMEOUT = -1, -6
DTYPE_F32, DTYPE_BF16 = 0, 1
ST_COMPUTE, ST_GIVEN = 0, 1
SCALES_ROWMAJOR, SCALES_MMA = 0, 1
(OP_QUANTIZE, OP_GEMM_W4A16, OP_GEMM_W4A4, OP_GROUPED_GEMM, OP_GATHER_ARGMAX, OP_GEMM_W4A4_QUANT,
 OP_GROUPED_GEMM_W4A4) = range(7)

EXPORTS = [
    "nvfp4_quantize", "nvfp4_prepack_scales", "nvfp4_gemm_w4a16", "nvfp4_gemm_w4a4",
    "nvfp4_moe_route", "nvfp4_grouped_gemm", "nvfp4_gather_gemv_argmax", "nvfp4_gather_rows", "nvfp4_gemv_argmax",
    "nvfp4_scales_bytes", "nvfp4_workspace_size", "nvfp4_status_string",
    "nvfp4_read_device_status", "nvfp4_selftest_bounded_wait", "nvfp4_version",
    "nvfp4_gemm_w4a16_noalloc", "nvfp4_verify_accept", "nvfp4_probe_fp4_mma_rate",
    "nvfp4_gemm_w4a16_silu_mul", "nvfp4_gemm_w4a4_quant", "nvfp4_grouped_gemm_w4a4",
]
_NON_INT = ("nvfp4_scales_bytes", "nvfp4_workspace_size", "nvfp4_status_string")


class CTensor(ctypes.Structure):
    """Mirror of nvfp4_tensor_t."""
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("s_t", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("K", ctypes.c_int64), ("batch", ctypes.c_int32),
                ("scale_layout", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libnvfp4.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(str(LIB_PATH))
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        L.nvfp4_quantize.argtypes = [vp, i32, i64, i64, vp, vp, vp, i32, i32, vp, sz, vp]
        L.nvfp4_prepack_scales.argtypes = [vp, i64, i64, i64, vp, vp]
        L.nvfp4_gemm_w4a16.argtypes = [vp, i64, CTensor, vp, vp, sz, vp]
        L.nvfp4_gemm_w4a4.argtypes = [CTensor, CTensor, vp, vp, sz, vp]
        L.nvfp4_gemm_w4a4_quant.argtypes = [CTensor, CTensor, vp, vp, vp, i32, vp, vp, sz, vp]
        L.nvfp4_gemm_w4a16_noalloc.argtypes = [vp, i64, CTensor, vp, vp]
        L.nvfp4_gemm_w4a16_silu_mul.argtypes = [vp, i64, CTensor, vp, vp, sz, vp]
        L.nvfp4_moe_route.argtypes = [vp, i64, i32, i32, vp, vp, vp]
        L.nvfp4_grouped_gemm.argtypes = [vp, i64, i32, vp, vp, CTensor, CTensor, vp, vp, sz, vp]
        L.nvfp4_grouped_gemm_w4a4.argtypes = [vp, i64, i32, vp, vp, CTensor, CTensor, vp, vp, sz, vp]
        L.nvfp4_gather_gemv_argmax.argtypes = [vp, i64, CTensor, vp, i64, vp, vp, vp, sz, vp]
        L.nvfp4_gather_rows.argtypes = [CTensor, vp, i64, vp, vp, vp]
        L.nvfp4_gemv_argmax.argtypes = [vp, i64, CTensor, vp, vp, vp, vp, sz, vp]
        L.nvfp4_verify_accept.argtypes = [vp, i64, i32, CTensor, vp, vp, vp, vp, sz, vp]
        L.nvfp4_scales_bytes.argtypes = [i64, i64, i32]
        L.nvfp4_scales_bytes.restype = sz
        L.nvfp4_workspace_size.argtypes = [i32, i64, i64, i64, i64, i64]
        L.nvfp4_workspace_size.restype = sz
        L.nvfp4_status_string.argtypes = [i32]
        L.nvfp4_status_string.restype = ctypes.c_char_p
        L.nvfp4_read_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), vp]
        L.nvfp4_selftest_bounded_wait.argtypes = [i64, vp]
        L.nvfp4_probe_fp4_mma_rate.argtypes = [i32, i32, vp]
        L.nvfp4_version.argtypes = []
        for name in EXPORTS:
            if name not in _NON_INT:
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != OK:
        raise RuntimeError(f"{what}: {lib().nvfp4_status_string(rc).decode()} ({rc})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise RuntimeError("nvfp4: tensors must live on a CUDA device (no CPU path exists)")


@dataclass
class QTensor:
    """An NVFP4 tensor on the device: codes uint8 [batch*rows][K/2], scales
    uint8 (row-major [batch*rows][K/16] or the MMA layout), s_t fp32 [batch]."""
    codes: torch.Tensor
    scales: torch.Tensor
    s_t: torch.Tensor
    rows: int
    K: int
    batch: int = 1
    scale_layout: int = SCALES_ROWMAJOR

    def c(self) -> CTensor:
        return CTensor(self.codes.data_ptr(), self.scales.data_ptr(), self.s_t.data_ptr(),
                       self.rows, self.K, self.batch, self.scale_layout)


def scales_bytes(rows: int, K: int, layout: int) -> int:
    return int(lib().nvfp4_scales_bytes(rows, K, layout))


def workspace_size(op: int, a=0, b=0, c=0, e=0, topk=0) -> int:
    return int(lib().nvfp4_workspace_size(op, a, b, c, e, topk))


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def quantize(x: torch.Tensor, s_t: torch.Tensor | None = None, scale_layout: int = SCALES_ROWMAJOR,
             workspace: torch.Tensor | None = None) -> QTensor:
    """NVFP4-quantise x [rows][K] (fp32 or bf16). s_t None -> computed from
    the tensor (amax / 2688); else a 1-element fp32 tensor to use."""
    _require_cuda(x)
    rows, K = x.shape
    dtype = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}[x.dtype]
    x = x.contiguous()
    codes = torch.empty(rows, K // 2, dtype=torch.uint8, device=x.device)
    scales = torch.empty(max(scales_bytes(rows, K, scale_layout), 1), dtype=torch.uint8, device=x.device)
    if s_t is None:
        st = torch.empty(1, dtype=torch.float32, device=x.device)
        mode = ST_COMPUTE
        ws = workspace if workspace is not None else _workspace(workspace_size(OP_QUANTIZE, rows, 0, K), x.device)
    else:
        st = s_t.to(device=x.device, dtype=torch.float32).reshape(1).contiguous()
        mode = ST_GIVEN
        ws = None
    _check(lib().nvfp4_quantize(_ptr(x), dtype, rows, K, _ptr(codes), _ptr(scales), _ptr(st), mode,
                                scale_layout, _ptr(ws), 0 if ws is None else ws.numel(), _stream()),
           "nvfp4_quantize")
    if scale_layout == SCALES_ROWMAJOR:
        scales = scales[: rows * (K // 16)].view(rows, K // 16)
    return QTensor(codes, scales, st, rows, K, 1, scale_layout)


def quantize_stack(mats) -> QTensor:
    """Quantise a list of equally shaped fp32/bf16 matrices (e.g. experts),
    each with its own tensor scale, into one batched QTensor (row-major)."""
    qs = [quantize(w) for w in mats]
    return QTensor(torch.cat([q.codes for q in qs]), torch.cat([q.scales for q in qs]),
                   torch.cat([q.s_t for q in qs]), qs[0].rows, qs[0].K, len(qs), SCALES_ROWMAJOR)


def prepack_scales(q: QTensor) -> QTensor:
    """Copy of q with its block scales re-laid into the MMA layout."""
    _require_cuda(q.codes)
    per = scales_bytes(q.rows, q.K, SCALES_MMA)
    dst = torch.empty(q.batch * per, dtype=torch.uint8, device=q.codes.device)
    _check(lib().nvfp4_prepack_scales(_ptr(q.scales), q.batch, q.rows, q.K, _ptr(dst), _stream()),
           "nvfp4_prepack_scales")
    return QTensor(q.codes, dst, q.s_t, q.rows, q.K, q.batch, SCALES_MMA)


def gemm_w4a16(x: torch.Tensor, w: QTensor, out: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Y = X @ W_hat^T, X bf16 [M][K], Y bf16 [M][N]."""
    _require_cuda(x)
    M = x.shape[0]
    y = out if out is not None else torch.empty(M, w.rows, dtype=torch.bfloat16, device=x.device)
    ws = workspace if workspace is not None else _workspace(workspace_size(OP_GEMM_W4A16, M, w.rows, w.K),
                                                            x.device)
    _check(lib().nvfp4_gemm_w4a16(_ptr(x), M, w.c(), _ptr(y), _ptr(ws), ws.numel(), _stream()),
           "nvfp4_gemm_w4a16")
    return y


def gemm_w4a16_silu_mul(x: torch.Tensor, w: QTensor, out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None) -> torch.Tensor:
    """h = bf16(silu(X @ W_gate^T) * (X @ W_up^T)); W stacks gate rows [0, I)
    and up rows [I, 2I). X bf16 [M][K] -> h bf16 [M][I]."""
    _require_cuda(x)
    M = x.shape[0]
    h = out if out is not None else torch.empty(M, w.rows // 2, dtype=torch.bfloat16, device=x.device)
    ws = workspace if workspace is not None else _workspace(workspace_size(OP_GEMM_W4A16, M, w.rows, w.K),
                                                            x.device)
    _check(lib().nvfp4_gemm_w4a16_silu_mul(_ptr(x), M, w.c(), _ptr(h), _ptr(ws), ws.numel(), _stream()),
           "nvfp4_gemm_w4a16_silu_mul")
    return h


def gemm_w4a4(a: QTensor, w: QTensor, out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Y = s_tA s_tW (A_q @ W_q^T) on the block-scaled FP4 tensor cores."""
    _require_cuda(a.codes)
    y = out if out is not None else torch.empty(a.rows, w.rows, dtype=torch.bfloat16, device=a.codes.device)
    ws = workspace if workspace is not None else _workspace(workspace_size(OP_GEMM_W4A4, a.rows, w.rows, a.K),
                                                            a.codes.device)
    _check(lib().nvfp4_gemm_w4a4(a.c(), w.c(), _ptr(y), _ptr(ws), ws.numel(), _stream()), "nvfp4_gemm_w4a4")
    return y


def gemm_w4a4_quant(a: QTensor, w: QTensor, s_t: torch.Tensor | None = None, y: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None) -> QTensor:
    """The W4A4 output as NVFP4 (MMA-layout scales), the next W4A4 layer's
    input. s_t given -> fused epilogue with that tensor scale; None -> the
    dynamic scale amax / 2688 (the bf16 output is written to `y` on the way)."""
    _require_cuda(a.codes)
    M, N = a.rows, w.rows
    dev = a.codes.device
    codes = torch.empty(M, N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(max(scales_bytes(M, N, SCALES_MMA), 1), dtype=torch.uint8, device=dev)
    if s_t is None:
        st = torch.empty(1, dtype=torch.float32, device=dev)
        mode = ST_COMPUTE
        y = y if y is not None else torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    else:
        st = s_t.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
        mode = ST_GIVEN
    ws = workspace if workspace is not None else _workspace(workspace_size(OP_GEMM_W4A4_QUANT, M, N, a.K), dev)
    _check(lib().nvfp4_gemm_w4a4_quant(a.c(), w.c(), _ptr(codes), _ptr(scales), _ptr(st), mode, _ptr(y), _ptr(ws),
                                       ws.numel(), _stream()), "nvfp4_gemm_w4a4_quant")
    return QTensor(codes, scales, st, M, N, 1, SCALES_MMA)


def moe_route(logits: torch.Tensor, topk: int):
    """ids int32 [T][topk], weights fp32 [T][topk] from fp32 router logits."""
    _require_cuda(logits)
    logits = logits.contiguous().float()
    T, E = logits.shape
    ids = torch.empty(T, topk, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, topk, dtype=torch.float32, device=logits.device)
    _check(lib().nvfp4_moe_route(_ptr(logits), T, E, topk, _ptr(ids), _ptr(w), _stream()), "nvfp4_moe_route")
    return ids, w


def grouped_gemm(x: torch.Tensor, ids: torch.Tensor, weights: torch.Tensor, w13: QTensor, w2: QTensor,
                 out: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Routed-expert MoE layer (gate/up + SiLU-mul + down + weighted combine)."""
    _require_cuda(x)
    T, H = x.shape
    topk = ids.shape[1]
    o = out if out is not None else torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    ws = workspace if workspace is not None else _workspace(
        workspace_size(OP_GROUPED_GEMM, T, H, w13.rows // 2, w13.batch, topk), x.device)
    _check(lib().nvfp4_grouped_gemm(_ptr(x), T, topk, _ptr(ids), _ptr(weights), w13.c(), w2.c(), _ptr(o),
                                    _ptr(ws), ws.numel(), _stream()), "nvfp4_grouped_gemm")
    return o


def grouped_gemm_w4a4(x: torch.Tensor, ids: torch.Tensor, weights: torch.Tensor, w13: QTensor, w2: QTensor,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Routed-expert MoE layer with NVFP4 activations (W4A4); w13 / w2 with
    MMA-layout scales (prepack_scales)."""
    _require_cuda(x)
    T, H = x.shape
    topk = ids.shape[1]
    o = out if out is not None else torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    ws = workspace if workspace is not None else _workspace(
        workspace_size(OP_GROUPED_GEMM_W4A4, T, H, w13.rows // 2, w13.batch, topk), x.device)
    _check(lib().nvfp4_grouped_gemm_w4a4(_ptr(x), T, topk, _ptr(ids), _ptr(weights), w13.c(), w2.c(), _ptr(o),
                                         _ptr(ws), ws.numel(), _stream()), "nvfp4_grouped_gemm_w4a4")
    return o


def gather_gemv_argmax(h: torch.Tensor, w: QTensor, idx: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None):
    """Masked draft head: (ids int32 [M], max logit fp32 [M])."""
    _require_cuda(h)
    M = h.shape[0]
    n_idx = w.rows if idx is None else idx.numel()
    ids = torch.empty(M, dtype=torch.int32, device=h.device)
    logit = torch.empty(M, dtype=torch.float32, device=h.device)
    ws = workspace if workspace is not None else _workspace(
        workspace_size(OP_GATHER_ARGMAX, M, n_idx, w.K), h.device)
    _check(lib().nvfp4_gather_gemv_argmax(_ptr(h), M, w.c(), _ptr(idx), n_idx, _ptr(ids), _ptr(logit),
                                          _ptr(ws), ws.numel(), _stream()), "nvfp4_gather_gemv_argmax")
    return ids, logit


def gather_rows(w: QTensor, idx: torch.Tensor) -> QTensor:
    """Compact NVFP4 copy of rows idx of w (one-time prepack of a fixed row subset)."""
    _require_cuda(w.codes, idx)
    n = idx.numel()
    codes = torch.empty(n, w.K // 2, dtype=torch.uint8, device=w.codes.device)
    scales = torch.empty(max(n * (w.K // 16), 1), dtype=torch.uint8, device=w.codes.device)
    _check(lib().nvfp4_gather_rows(w.c(), _ptr(idx), n, _ptr(codes), _ptr(scales), _stream()), "nvfp4_gather_rows")
    return QTensor(codes, scales, w.s_t, n, w.K)


def gemv_argmax(h: torch.Tensor, w: QTensor, ids: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None):
    """Argmax over all rows of w, row j reported as ids[j]: (ids int32 [M], max logit fp32 [M])."""
    _require_cuda(h)
    M = h.shape[0]
    out = torch.empty(M, dtype=torch.int32, device=h.device)
    logit = torch.empty(M, dtype=torch.float32, device=h.device)
    ws = workspace if workspace is not None else _workspace(
        workspace_size(OP_GATHER_ARGMAX, M, w.rows, w.K), h.device)
    _check(lib().nvfp4_gemv_argmax(_ptr(h), M, w.c(), _ptr(ids), _ptr(out), _ptr(logit), _ptr(ws), ws.numel(),
                                   _stream()), "nvfp4_gemv_argmax")
    return out, logit


def verify_accept(h: torch.Tensor, w: QTensor, draft_ids: torch.Tensor, workspace: torch.Tensor | None = None):
    """Speculative verify: h bf16 [batch * (n_draft + 1)][K], draft_ids int32
    [batch][n_draft] -> (argmax ids int32 [batch][n_draft + 1], accepted
    drafts int32 [batch])."""
    _require_cuda(h, draft_ids)
    batch, n_draft = draft_ids.shape
    if h.shape[0] != batch * (n_draft + 1):
        raise ValueError("verify_accept: h needs batch * (n_draft + 1) rows")
    draft_ids = draft_ids.to(torch.int32).contiguous()
    tokens = torch.empty(batch, n_draft + 1, dtype=torch.int32, device=h.device)
    n_acc = torch.empty(batch, dtype=torch.int32, device=h.device)
    ws = workspace if workspace is not None else _workspace(
        workspace_size(OP_GATHER_ARGMAX, h.shape[0], w.rows, w.K), h.device)
    _check(lib().nvfp4_verify_accept(_ptr(h), batch, n_draft, w.c(), _ptr(draft_ids), _ptr(tokens), _ptr(n_acc),
                                     _ptr(ws), ws.numel(), _stream()), "nvfp4_verify_accept")
    return tokens, n_acc


def read_device_status() -> int:
    v = ctypes.c_int(0)
    _check(lib().nvfp4_read_device_status(ctypes.byref(v), _stream()), "nvfp4_read_device_status")
    return v.value


def probe_fp4_mma_rate(n_mma: int, n_ctas: int = 0) -> None:
    """Launch the FP4 tensor-core issue-rate probe on the current stream."""
    _check(lib().nvfp4_probe_fp4_mma_rate(n_mma, n_ctas, _stream()), "nvfp4_probe_fp4_mma_rate")


def selftest_bounded_wait(limit_ns: int) -> None:
    _check(lib().nvfp4_selftest_bounded_wait(limit_ns, _stream()), "nvfp4_selftest_bounded_wait")
