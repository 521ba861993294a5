"""The oracle's quantisation of a stack of expert matrices, spread over
spawned worker processes (each expert is quantised by oracle.quantize with
its own tensor scale, as in the layer's definition). Test infrastructure
only: it calls the oracle and nothing of the CUDA path."""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def _quantize_one(w):
    import oracle as O
    q = O.quantize(w)
    return q.codes, q.scales, q.s_t


def quantize_experts(mats, workers: int | None = None):
    """[oracle.QTensor] for fp32 matrices `mats` (e.g. [E][2I][H])."""
    import oracle as O
    mats = [np.ascontiguousarray(np.asarray(m, dtype=np.float32)) for m in mats]
    n = workers or max(1, min(os.cpu_count() or 1, 16, len(mats)))
    with ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
        return [O.QTensor(c, s, st) for c, s, st in ex.map(_quantize_one, mats)]
