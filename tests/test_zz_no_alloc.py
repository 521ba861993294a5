"""The allocation-free W4A16 entry point, for callers that cannot allocate
device memory on their decode path (an engine that has reserved almost all
device memory for its KV cache, or a host that must not call cudaMalloc /
cudaFree there because they can synchronise the device).

Calls nvfp4_gemm_w4a16_noalloc through the C ABI and checks its output
against nvfp4_gemm_w4a16 (which takes a caller workspace) on two calls in a
row with different inputs, so a stale library scratch would show. This file
is collected last on purpose; it passes alone or after the other tests."""
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


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    nv, L = _lib()
    dev = torch.device("cuda:0")
    N, K = 1000, 2048
    w = synth.normal_f32((N, K), 0.02, seed=51).to(dev)
    q = nv.quantize(w)
    for call, M in enumerate((32, 5)):
        x = synth.normal_bf16((M, K), seed=52 + call).to(dev)
        y_ref = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(nv.workspace_size(nv.OP_GEMM_W4A16, M, N, K), dtype=torch.uint8, device=dev)
        rc = L.nvfp4_gemm_w4a16(ctypes.c_void_p(x.data_ptr()), M, q.c(), ctypes.c_void_p(y_ref.data_ptr()),
                                ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream())
        assert rc == 0
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        rc = L.nvfp4_gemm_w4a16_noalloc(ctypes.c_void_p(x.data_ptr()), M, q.c(), ctypes.c_void_p(y.data_ptr()),
                                        _stream())
        assert rc == 0
        torch.cuda.synchronize()
        a = y.float().cpu().numpy().astype(np.float64)
        b = y_ref.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(a))
        assert O.rel_fro(a, b) <= TOL, (call, O.rel_fro(a, b))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    nv, L = _lib()
    dev = torch.device("cuda:0")
    for M, K in ((33, 256), (4, 32768 + 128)):
        q = nv.quantize(synth.normal_f32((64, K), 0.02, seed=53).to(dev))
        x = torch.zeros(M, K, dtype=torch.bfloat16, device=dev)
        y = torch.zeros(M, 64, dtype=torch.bfloat16, device=dev)
        rc = L.nvfp4_gemm_w4a16_noalloc(ctypes.c_void_p(x.data_ptr()), M, q.c(), ctypes.c_void_p(y.data_ptr()),
                                        _stream())
        assert rc == -7
        assert "scratch" in L.nvfp4_status_string(rc).decode()
