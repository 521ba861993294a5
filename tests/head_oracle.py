"""The oracle's logits over every row of the 248,320 x 5120 draft head.

The oracle takes about 12 s per 8192 rows on one core, so the rows are split
into the seeded blocks of synth.draft_head_block and handed to a pool of
spawned worker processes: each redraws its block, quantises it with the whole
head's tensor scale (oracle.quantize, s_t given) and takes fp64 dot products
with the hidden states. Test infrastructure only: it calls the oracle and the
seeded generators and nothing of the CUDA path."""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def _block_logits(args):
    b, st, h = args
    import oracle as O
    import synth
    q = O.quantize(synth.draft_head_block(b).numpy(), s_t=st)
    return b, np.asarray(h, dtype=np.float64) @ O.decode(q).T


def full_head_logits(h, s_t, workers: int | None = None):
    """fp64 logits [len(h)][V] of hidden states h (fp32/fp64 [M][K]) against
    every head row, rows quantised with tensor scale s_t."""
    import synth
    nb = synth.draft_head_blocks()
    h = np.asarray(h, dtype=np.float64)
    out = np.empty((h.shape[0], synth.VOCAB), dtype=np.float64)
    n = workers or max(1, min(os.cpu_count() or 1, 16, nb))
    # spawned (not forked) workers: the parent may already hold a CUDA context;
    # a worker that dies raises BrokenProcessPool here instead of hanging
    with ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
        for b, lg in ex.map(_block_logits, [(b, s_t, h) for b in range(nb)]):
            r0 = b * synth.HEAD_BLOCK
            out[:, r0:r0 + lg.shape[1]] = lg
    return out
