"""Shared helpers of the GPU parity tests (the CUDA path through the C ABI,
compared with the CPU oracle on the same seeded inputs)."""
import numpy as np
import torch

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def nv():
    import nvfp4_block_scaled_04_gb300 as m
    m.lib()
    return m


def np_u8(t):
    return t.detach().cpu().numpy().astype(np.uint8)


def np_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def unpack_mma_scales(buf, rows, K):
    """Read row-major [rows][K/16] block scales back out of the MMA layout
    (the layout formula of include/nvfp4.h, written out independently)."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    kc = K // 16
    cols4 = (kc + 3) // 4 * 4
    r = np.arange(rows)[:, None]
    c = np.arange(kc)[None, :]
    off = ((r // 128) * (cols4 // 4) + c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4
    return buf[off]
