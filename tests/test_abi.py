"""CPU-side checks of the C ABI: the library builds, loads without a GPU,
exports every entry point include/nvfp4.h declares, and its host-only helpers
(sizes, status strings, argument validation) behave. No kernel is launched."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "nvfp4.h"


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_04_gb300 as nv
    if not nv.LIB_PATH.exists():
        from nvfp4_block_scaled_04_gb300 import _build
        _build.build()
    nv.lib()
    return nv


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(nvfp4_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for f in ["nvfp4_quantize", "nvfp4_gemm_w4a16", "nvfp4_gemm_w4a4", "nvfp4_grouped_gemm",
              "nvfp4_gather_gemv_argmax"]:
        assert f in names


def test_library_exports_every_declared_symbol(nv):
    L = nv.lib()
    missing = [f for f in declared_functions() if not hasattr(L, f)]
    assert not missing, missing
    assert set(declared_functions()) == set(nv.EXPORTS)


def test_status_strings(nv):
    L = nv.lib()
    for code in range(0, -7, -1):
        s = L.nvfp4_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.nvfp4_status_string(-99).decode() == "unknown status"


def test_scale_bytes(nv):
    assert nv.scales_bytes(300, 320, nv.SCALES_ROWMAJOR) == 300 * 20
    # MMA layout pads rows to 128 and scale columns to 4
    assert nv.scales_bytes(300, 320, nv.SCALES_MMA) == 384 * 20
    assert nv.scales_bytes(128, 64 * 3 + 16, nv.SCALES_MMA) == 128 * 16
    assert nv.scales_bytes(8192, 5120, nv.SCALES_MMA) == 8192 * 320


def test_workspace_sizes_grow_with_the_problem(nv):
    a = nv.workspace_size(nv.OP_GEMM_W4A16, 1, 34816, 5120)
    b = nv.workspace_size(nv.OP_GEMM_W4A16, 32, 34816, 5120)
    assert 0 < a <= b
    assert nv.workspace_size(nv.OP_GEMM_W4A16, 33, 1, 5120) > b
    assert nv.workspace_size(nv.OP_GROUPED_GEMM, 4096, 2048, 768, 128, 8) > \
        nv.workspace_size(nv.OP_GROUPED_GEMM, 256, 2048, 768, 128, 8) > 0
    assert nv.workspace_size(nv.OP_GATHER_ARGMAX, 8, 32768, 5120) > 0
    assert nv.workspace_size(nv.OP_QUANTIZE, 10, 0, 64) >= 4
    assert nv.workspace_size(nv.OP_GEMM_W4A4, 8192, 34816, 5120) == 8192 * 320 + 34816 * 320


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_validation_rejects_before_launch(nv):
    L = nv.lib()
    ws = _fake(0x20000)
    # K not a multiple of 16
    assert L.nvfp4_quantize(_fake(), nv.DTYPE_BF16, 4, 40, _fake(), _fake(), _fake(), nv.ST_COMPUTE,
                            nv.SCALES_ROWMAJOR, ws, 256, None) == -2
    # bad dtype / mode / layout
    assert L.nvfp4_quantize(_fake(), 7, 4, 64, _fake(), _fake(), _fake(), 0, 0, ws, 256, None) == -1
    assert L.nvfp4_quantize(_fake(), 1, 4, 64, _fake(), _fake(), _fake(), 5, 0, ws, 256, None) == -1
    assert L.nvfp4_quantize(_fake(), 1, 4, 64, _fake(), _fake(), _fake(), 0, 9, ws, 256, None) == -1
    # misaligned input
    assert L.nvfp4_quantize(_fake(0x10001), 1, 4, 64, _fake(), _fake(), _fake(), 0, 0, ws, 256, None) == -3
    # missing workspace in COMPUTE mode
    assert L.nvfp4_quantize(_fake(), 1, 4, 64, _fake(), _fake(), _fake(), 0, 0, None, 0, None) == -5
    W = nv.CTensor(0x30000, 0x40000, 0x50000, 256, 100, 1, 0)
    assert L.nvfp4_gemm_w4a16(_fake(), 4, W, _fake(), ws, 1 << 20, None) == -2       # K % 128
    W = nv.CTensor(0x30000, 0x40000, 0x50000, 256, 256, 1, 1)
    assert L.nvfp4_gemm_w4a16(_fake(), 4, W, _fake(), ws, 1 << 20, None) == -1       # MMA scales
    W = nv.CTensor(0x30000, 0x40000, 0x50000, 256, 256, 1, 0)
    assert L.nvfp4_gemm_w4a16(_fake(), 4, W, _fake(), None, 0, None) == -5            # workspace
    A = nv.CTensor(0x30000, 0x40000, 0x50000, 64, 96, 1, 1)
    assert L.nvfp4_gemm_w4a4(A, A, _fake(), ws, 1 << 20, None) == -2                 # K % 64
    B = nv.CTensor(0x30000, 0x40000, 0x50000, 64, 128, 1, 1)
    C = nv.CTensor(0x30000, 0x40000, 0x50000, 64, 256, 1, 1)
    assert L.nvfp4_gemm_w4a4(B, C, _fake(), ws, 1 << 20, None) == -1                 # K mismatch
    D = nv.CTensor(0x30000, 0x40000, 0x50000, 60, 128, 1, 1)
    assert L.nvfp4_gemm_w4a4(B, D, _fake(), ws, 1 << 20, None) == -2                 # N % 8
    Brm = nv.CTensor(0x30000, 0x40000, 0x50000, 64, 128, 1, 0)
    assert L.nvfp4_gemm_w4a4(Brm, B, _fake(), None, 0, None) == -5                   # relayout ws
    assert L.nvfp4_gather_gemv_argmax(_fake(), 33, W, None, 0, _fake(), None, ws, 1 << 20, None) == -1
    assert L.nvfp4_moe_route(_fake(), 4, 2000, 8, _fake(), _fake(), None) == -1
    W13 = nv.CTensor(0x30000, 0x40000, 0x50000, 256, 128, 4, 0)
    W2 = nv.CTensor(0x30000, 0x40000, 0x50000, 128, 256, 3, 0)                      # batch mismatch
    assert L.nvfp4_grouped_gemm(_fake(), 4, 2, _fake(), _fake(), W13, W2, _fake(), ws, 1 << 30, None) == -1
    assert L.nvfp4_selftest_bounded_wait(0, None) == -1


def test_row_gather_and_compact_argmax_validate_arguments(nv):
    L = nv.lib()
    ws = _fake()
    W = nv.CTensor(0x1000, 0x2000, 0x3000, 64, 256, 1, 0)
    assert L.nvfp4_gather_rows(W, None, 4, _fake(), _fake(), None) == -1             # no index
    Wk = nv.CTensor(0x1000, 0x2000, 0x3000, 64, 48, 1, 0)
    assert L.nvfp4_gather_rows(Wk, _fake(), 4, _fake(), _fake(), None) == -2         # K % 32
    assert L.nvfp4_gemv_argmax(_fake(), 0, W, None, _fake(), None, ws, 1 << 20, None) == -1   # M
    Wa = nv.CTensor(0x1000, 0x2000, 0x3000, 64, 384, 1, 0)
    assert L.nvfp4_gemv_argmax(_fake(), 1, Wa, None, _fake(), None, ws, 1 << 20, None) == -2  # K % 256
    assert L.nvfp4_gemv_argmax(_fake(), 1, W, None, _fake(), None, None, 0, None) == -5       # workspace


def test_verify_accept_validates_arguments(nv):
    L = nv.lib()
    ws = _fake()
    W = nv.CTensor(0x1000, 0x2000, 0x3000, 64, 256, 1, 0)
    ok = (_fake(), 4, 3, W, _fake(), _fake(), _fake(), ws, 1 << 20, None)
    assert L.nvfp4_verify_accept(_fake(), 9, 3, W, _fake(), _fake(), _fake(), ws, 1 << 20, None) == -1  # 36 rows
    assert L.nvfp4_verify_accept(_fake(), 4, 3, W, None, _fake(), _fake(), ws, 1 << 20, None) == -1    # no drafts
    assert L.nvfp4_verify_accept(_fake(), 0, 3, W, _fake(), _fake(), _fake(), ws, 1 << 20, None) == -1  # batch
    Wa = nv.CTensor(0x1000, 0x2000, 0x3000, 64, 384, 1, 0)
    assert L.nvfp4_verify_accept(_fake(), 4, 3, Wa, _fake(), _fake(), _fake(), ws, 1 << 20, None) == -2  # K % 256
    assert L.nvfp4_verify_accept(_fake(0x1008), *ok[1:]) == -3                                          # H misaligned
    assert L.nvfp4_verify_accept(*ok[:7], None, 0, None) == -5                                          # workspace


def test_grouped_gemm_validates_arguments(nv):
    L = nv.lib()
    ws = _fake(0x20000)
    E, H, I = 4, 256, 256
    W13 = nv.CTensor(0x30000, 0x40000, 0x50000, 2 * I, H, E, 0)
    W2 = nv.CTensor(0x60000, 0x70000, 0x80000, H, I, E, 0)
    need = nv.workspace_size(nv.OP_GROUPED_GEMM, 64, H, I, E, 2)
    args = (_fake(), 64, 2, _fake(), _fake())
    assert L.nvfp4_grouped_gemm(*args, W13, W2, _fake(), ws, need - 1, None) == -5          # workspace short
    assert L.nvfp4_grouped_gemm(*args, W13, W2, _fake(), None, 0, None) == -5               # no workspace
    assert L.nvfp4_grouped_gemm(_fake(0x10008), 64, 2, _fake(), _fake(), W13, W2, _fake(), ws, need,
                                None) == -3                                                  # X misaligned
    assert L.nvfp4_grouped_gemm(_fake(), 64, 5, _fake(), _fake(), W13, W2, _fake(), ws, 1 << 30,
                                None) == -1                                                  # topk > E
    assert L.nvfp4_grouped_gemm(_fake(), 64, 0, _fake(), _fake(), W13, W2, _fake(), ws, 1 << 30,
                                None) == -1                                                  # topk < 1
    W13m = nv.CTensor(0x30000, 0x40000, 0x50000, 2 * I, H, E, 1)
    assert L.nvfp4_grouped_gemm(*args, W13m, W2, _fake(), ws, 1 << 30, None) == -1          # MMA scales
    W13k = nv.CTensor(0x30000, 0x40000, 0x50000, 2 * I, 192, E, 0)
    W2k = nv.CTensor(0x60000, 0x70000, 0x80000, 192, I, E, 0)
    assert L.nvfp4_grouped_gemm(*args, W13k, W2k, _fake(), ws, 1 << 30, None) == -2        # H % 128
    assert L.nvfp4_grouped_gemm(_fake(), 0, 2, _fake(), _fake(), W13, W2, _fake(), None, 0, None) == 0   # T = 0


def test_grouped_workspace_holds_the_tile_table(nv):
    """The tensor-core tile table (up to 128 routed rows of one expert per
    tile) grows the workspace with T and E, in steps of whole tables."""
    H, I = 2048, 768
    small = nv.workspace_size(nv.OP_GROUPED_GEMM, 4096, H, I, 128, 8)
    more_experts = nv.workspace_size(nv.OP_GROUPED_GEMM, 4096, H, I, 256, 8)
    assert more_experts > small
    assert nv.workspace_size(nv.OP_GROUPED_GEMM, 4096 + 16, H, I, 128, 8) > small


def test_grouped_gemm_w4a4_validates_arguments(nv):
    L = nv.lib()
    ws = _fake(0x20000)
    E, H, I = 4, 256, 128
    W13 = nv.CTensor(0x30000, 0x40000, 0x50000, 2 * I, H, E, 1)
    W2 = nv.CTensor(0x60000, 0x70000, 0x80000, H, I, E, 1)
    need = nv.workspace_size(nv.OP_GROUPED_GEMM_W4A4, 64, H, I, E, 2)
    assert need > nv.workspace_size(nv.OP_GROUPED_GEMM_W4A4, 16, H, I, E, 2)
    args = (_fake(), 64, 2, _fake(), _fake())
    W13r = nv.CTensor(0x30000, 0x40000, 0x50000, 2 * I, H, E, 0)
    assert L.nvfp4_grouped_gemm_w4a4(*args, W13r, W2, _fake(), ws, need, None) == -1          # row-major scales
    W13h = nv.CTensor(0x30000, 0x40000, 0x50000, 2 * I, 128, E, 1)
    W2h = nv.CTensor(0x60000, 0x70000, 0x80000, 128, I, E, 1)
    assert L.nvfp4_grouped_gemm_w4a4(*args, W13h, W2h, _fake(), ws, need, None) == -2         # H % 256
    assert L.nvfp4_grouped_gemm_w4a4(*args, W13, W2, _fake(), ws, need - 1, None) == -5       # workspace
    W13s = nv.CTensor(0x30000, 0x40008, 0x50000, 2 * I, H, E, 1)
    assert L.nvfp4_grouped_gemm_w4a4(*args, W13s, W2, _fake(), ws, need, None) == -3          # scales misaligned
    assert L.nvfp4_grouped_gemm_w4a4(_fake(), 0, 2, _fake(), _fake(), W13, W2, _fake(), None, 0, None) == 0


def test_w4a4_quant_validates_arguments(nv):
    L = nv.lib()
    ws = _fake(0x20000)
    A = nv.CTensor(0x30000, 0x40000, 0x50000, 256, 512, 1, 1)
    W = nv.CTensor(0x60000, 0x70000, 0x80000, 256, 512, 1, 1)
    Wn = nv.CTensor(0x60000, 0x70000, 0x80000, 200, 512, 1, 1)
    need = nv.workspace_size(nv.OP_GEMM_W4A4_QUANT, 256, 256, 512)
    assert need >= 256
    f = _fake
    assert L.nvfp4_gemm_w4a4_quant(A, Wn, f(), f(), f(), 1, None, ws, need, None) == -2   # N % 64
    assert L.nvfp4_gemm_w4a4_quant(A, W, f(), f(), f(), 0, None, ws, need, None) == -1    # COMPUTE needs Y
    assert L.nvfp4_gemm_w4a4_quant(A, W, f(), f(), f(), 3, None, ws, need, None) == -1    # bad mode
    assert L.nvfp4_gemm_w4a4_quant(A, W, f(0x1008), f(), f(), 1, None, ws, need, None) == -3   # codes misaligned
    assert L.nvfp4_gemm_w4a4_quant(A, W, f(), f(), f(), 1, None, ws, need - 1, None) == -5     # workspace
