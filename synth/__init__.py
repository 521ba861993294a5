"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests
and the benchmark.

This module draws random numbers and nothing else: it holds none of the NVFP4
arithmetic (no scaling, rounding, encoding or matmul), so that the oracle and
the CUDA path can both consume its tensors without sharing any of the method.

Every draw uses its own ``torch.Generator`` seeded explicitly, on the CPU, so
the same seed gives the same tensor on every machine and in every process.
Shapes follow the workloads the pages serve: a ~27B dense decoder (hidden
5120, fused gate/up 34816, down 17408 -> 5120), a 248,320-entry vocabulary
with a 32,768-id draft mask ("The masked head trick"), and a 35B-A3B style
MoE layer (128 experts, top-8, hidden 2048, expert intermediate 768).
"""
from __future__ import annotations

import torch

# --- layer shapes of the served models -------------------------------------
HIDDEN_27B = 5120
GATE_UP_27B = 34816          # fused gate+up output features
INTER_27B = 17408            # down-projection input features
VOCAB = 248320
MASK_ROWS = 32768
MOE_EXPERTS = 128
MOE_TOPK = 8
MOE_HIDDEN = 2048
MOE_INTER = 768


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_f32(shape, std: float, seed: int) -> torch.Tensor:
    """fp32 N(0, std^2) on the CPU."""
    return torch.randn(*shape, generator=_gen(seed), dtype=torch.float32) * std


def normal_bf16(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    """bf16 N(0, std^2): drawn in fp32, then rounded to nearest-even bf16."""
    return (torch.randn(*shape, generator=_gen(seed), dtype=torch.float32) * std).to(torch.bfloat16)


def student_t_bf16(shape, df: int, seed: int) -> torch.Tensor:
    """bf16 Student-t(df) for integer df: Z / sqrt(chi2_df / df), chi2 as a sum
    of df squared standard normals, all from one seeded generator."""
    g = _gen(seed)
    z = torch.randn(*shape, generator=g, dtype=torch.float64)
    chi2 = torch.zeros(*shape, dtype=torch.float64)
    for _ in range(int(df)):
        chi2 += torch.randn(*shape, generator=g, dtype=torch.float64) ** 2
    t = z / torch.sqrt(chi2 / df)
    return t.to(torch.float32).to(torch.bfloat16)


def permutation_prefix(n: int, k: int, seed: int) -> torch.Tensor:
    """int32 ids: the first k entries of a seeded permutation of range(n)."""
    return torch.randperm(n, generator=_gen(seed))[:k].to(torch.int32)


def uniform_int(shape, lo: int, hi: int, seed: int) -> torch.Tensor:
    """int64 uniform in [lo, hi)."""
    return torch.randint(lo, hi, tuple(shape), generator=_gen(seed))


# --- per-workload recipes (seeds fixed so every consumer sees the same data) --

def tiny_w4a16(seed: int = 0):
    """M=4, K=256, N=512: weights fp32 N(0, 0.02^2), activations bf16 N(0,1)."""
    g = _gen(seed)
    w = torch.randn(512, 256, generator=g, dtype=torch.float32) * 0.02
    x = torch.randn(4, 256, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return w, x


def decode_weight(which: str) -> torch.Tensor:
    """27B-shaped decode weights: 'gate_up' [34816][5120] (seed 0) or
    'down' [5120][17408] (seed 1), fp32 N(0, 0.02^2)."""
    if which == "gate_up":
        return normal_f32((GATE_UP_27B, HIDDEN_27B), 0.02, seed=0)
    if which == "down":
        return normal_f32((HIDDEN_27B, INTER_27B), 0.02, seed=1)
    raise ValueError(which)


def decode_activation(M: int, K: int) -> torch.Tensor:
    """bf16 N(0,1) decode activations [M][K], seed 2 + M."""
    return normal_bf16((M, K), seed=2 + M)


def prefill_inputs(M: int = 8192, K: int = HIDDEN_27B, N: int = GATE_UP_27B):
    """W4A4 prefill: activations bf16 Student-t(4) [M][K] (seed 3), weights
    fp32 N(0, 0.02^2) [N][K] (seed 4)."""
    return student_t_bf16((M, K), 4, seed=3), normal_f32((N, K), 0.02, seed=4)


HEAD_BLOCK = 4096            # rows of the draft head drawn per seed


def draft_head_blocks(V: int = VOCAB) -> int:
    return (V + HEAD_BLOCK - 1) // HEAD_BLOCK


def draft_head_block(b: int, V: int = VOCAB, K: int = HIDDEN_27B) -> torch.Tensor:
    """Rows [4096 b, min(4096 (b + 1), V)) of the LM-head weight, fp32
    N(0, 0.02^2), seed 5_000_000 + b: every block has its own generator, so a
    worker process can redraw any block without the others."""
    r0 = b * HEAD_BLOCK
    return normal_f32((min(HEAD_BLOCK, V - r0), K), 0.02, seed=5_000_000 + b)


def draft_head_weight(V: int = VOCAB, K: int = HIDDEN_27B) -> torch.Tensor:
    """LM-head weight fp32 N(0, 0.02^2) [V][K]: the blocks of draft_head_block."""
    return torch.cat([draft_head_block(b, V, K) for b in range(draft_head_blocks(V))])


def draft_mask(V: int = VOCAB, n: int = MASK_ROWS) -> torch.Tensor:
    """The masked-vocabulary ids: first n of a seeded permutation (seed 6)."""
    return permutation_prefix(V, n, seed=6)


def draft_hidden(M: int, step: int, K: int = HIDDEN_27B) -> torch.Tensor:
    """bf16 N(0,1) draft-head hidden states [M][K] for draft step `step`."""
    return normal_bf16((M, K), seed=7 + step)


def verify_hidden(M: int = 32, K: int = HIDDEN_27B) -> torch.Tensor:
    """bf16 N(0,1) hidden states of a speculative verify batch [M][K] (seed 20):
    batch x (drafts + 1) positions, at most 32 rows."""
    return normal_bf16((M, K), seed=20)


def moe_inputs(T: int, E: int = MOE_EXPERTS, H: int = MOE_HIDDEN, I: int = MOE_INTER):
    """MoE layer: router logits fp32 N(0,1) [T][E] (seed 8), tokens bf16 N(0,1)
    [T][H] (seed 9), W13 fp32 N(0,0.02^2) [E][2I][H] (seed 10), W2 [E][H][I]
    (seed 11)."""
    logits = normal_f32((T, E), 1.0, seed=8)
    x = normal_bf16((T, H), seed=9)
    w13 = normal_f32((E, 2 * I, H), 0.02, seed=10)
    w2 = normal_f32((E, H, I), 0.02, seed=11)
    return logits, x, w13, w2
