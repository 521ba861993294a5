"""The allocation-free W4A16 entry point, for callers that cannot allocate
device memory on their decode path (an engine that has reserved almost all
device memory for its KV cache, or a host that must not call cudaMalloc /
cudaFree there because they can synchronise the device).

Calls nvfp4_gemm_w4a16_noalloc through the C ABI and checks its output
against the oracle (sampled output columns, recomputed in fp64 from the
oracle's own quantisation) and against nvfp4_gemm_w4a16 (which takes a caller
workspace), on two calls in a row with different inputs, so a stale library
scratch would show. Shapes: a small ragged one, the 27B down projection
(17408 -> 5120, split along K across CTAs), the documented maximum (32 tokens,
K = 32768, the split-K partials filling most of the fixed array) and K = 384
(the register-fed kernel). This file is collected last on purpose; it passes
alone or after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _lib():
    import nvfp4_block_scaled_04_gb300 as nv
    return nv, nv.lib()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(L, x, M, q, y):
    return L.nvfp4_gemm_w4a16_noalloc(ctypes.c_void_p(x.data_ptr()), M, q.c(), ctypes.c_void_p(y.data_ptr()),
                                      _stream())


@pytest.mark.parametrize("N,K,Ms", [(1000, 2048, (32, 5)), (5120, 17408, (1, 32)), (4864, 32768, (32, 3)),
                                    (300, 384, (7, 32))])
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls(N, K, Ms):
    nv, L = _lib()
    dev = torch.device("cuda:0")
    w = synth.normal_f32((N, K), 0.02, seed=51 + K)
    q = nv.quantize(w.to(dev))
    # the oracle on 192 sampled output columns, quantised with the whole tensor's scale
    cols = np.sort(np.random.default_rng(K).choice(N, min(N, 192), replace=False))
    wq_ref = O.quantize(w.numpy()[cols], s_t=O.tensor_scale(w.numpy()))
    del w
    for call, M in enumerate(Ms):
        x = synth.normal_bf16((M, K), seed=52 + call + K).to(dev)
        y_ref = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(nv.workspace_size(nv.OP_GEMM_W4A16, M, N, K), dtype=torch.uint8, device=dev)
        rc = L.nvfp4_gemm_w4a16(ctypes.c_void_p(x.data_ptr()), M, q.c(), ctypes.c_void_p(y_ref.data_ptr()),
                                ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream())
        assert rc == 0
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        assert _noalloc(L, x, M, q, y) == 0
        torch.cuda.synchronize()
        a = y.float().cpu().numpy().astype(np.float64)
        b = y_ref.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(a))
        assert O.rel_fro(a, b) <= TOL, (call, O.rel_fro(a, b))
        ref = O.gemm_w4a16(x.float().cpu().numpy(), wq_ref)
        assert O.rel_fro(a[:, cols], ref) <= TOL, (call, O.rel_fro(a[:, cols], ref))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    nv, L = _lib()
    dev = torch.device("cuda:0")
    for M, K in ((33, 256), (4, 32768 + 128)):
        q = nv.quantize(synth.normal_f32((64, K), 0.02, seed=53).to(dev))
        x = torch.zeros(M, K, dtype=torch.bfloat16, device=dev)
        y = torch.zeros(M, 64, dtype=torch.bfloat16, device=dev)
        rc = _noalloc(L, x, M, q, y)
        assert rc == -7
        assert "scratch" in L.nvfp4_status_string(rc).decode()
