"""Masked draft head (gathered-row GEMV + argmax) against the oracle."""
import functools

import numpy as np
import pytest
import torch

import oracle as O
import synth
from tests.gpu_common import DEV, nv

pytestmark = pytest.mark.gpu
TOL = 1e-2


def check_against_oracle(ids, logit, h, wq_ref, idx):
    oid, omax, logits = O.gather_gemv_argmax(h, wq_ref, idx)
    margin = O.top2_margin(logits)
    for m in range(len(ids)):
        rows = np.arange(wq_ref.codes.shape[0]) if idx is None else np.asarray(idx)
        assert int(ids[m]) in set(rows.tolist())
        if margin[m] > TOL:
            assert int(ids[m]) == int(oid[m]), (m, margin[m])
        else:   # near-tie: either of the top two is fine, and the value must match
            top2 = rows[np.argsort(logits[m])[-2:]]
            assert int(ids[m]) in set(top2.tolist())
        assert abs(float(logit[m]) - omax[m]) <= TOL * np.sqrt(np.mean(logits[m] ** 2))


@pytest.mark.parametrize("M", [1, 3, 4, 8, 32])
@pytest.mark.parametrize("masked", [True, False])
def test_small_head(M, masked):
    m = nv()
    V, K = 3000, 512
    w = synth.normal_f32((V, K), 0.02, seed=21)
    idx = synth.permutation_prefix(V, 700, seed=22) if masked else None
    h = synth.normal_bf16((M, K), seed=23 + M)
    ids, logit = m.gather_gemv_argmax(h.to(DEV), m.quantize(w.to(DEV)), None if idx is None else idx.to(DEV))
    check_against_oracle(ids.cpu().numpy(), logit.cpu().numpy(), h.float().numpy(), O.quantize(w.numpy()),
                         None if idx is None else idx.numpy())


def test_identity_index_equals_full_and_repeat_calls_agree():
    m = nv()
    V, K = 1000, 256
    w = m.quantize(synth.normal_f32((V, K), 0.02, seed=31).to(DEV))
    h = synth.normal_bf16((4, K), seed=32).to(DEV)
    ws = torch.zeros(m.workspace_size(m.OP_GATHER_ARGMAX, 4, V, K), dtype=torch.uint8, device=DEV)
    a = m.gather_gemv_argmax(h, w, None, workspace=ws)
    b = m.gather_gemv_argmax(h, w, torch.arange(V, dtype=torch.int32, device=DEV), workspace=ws)
    c = m.gather_gemv_argmax(h, w, None, workspace=ws)
    assert torch.equal(a[0], b[0]) and torch.equal(a[0], c[0]) and torch.equal(a[1], c[1])


def test_planted_winner():
    m = nv()
    V, K = 5000, 256
    w = synth.normal_f32((V, K), 0.02, seed=41)
    h = synth.normal_bf16((1, K), seed=42)
    idx = synth.permutation_prefix(V, 900, seed=43)
    target = int(idx[600])
    w[target] = torch.sign(h[0].float()) * 0.05
    ids, _ = m.gather_gemv_argmax(h.to(DEV), m.quantize(w.to(DEV)), idx.to(DEV))
    assert int(ids[0]) == target


@functools.lru_cache(maxsize=1)
def _head():
    """(fp32 head, mask, GPU quantisation, oracle tensor scale, oracle masked rows)."""
    w = synth.draft_head_weight()
    idx = synth.draft_mask()
    st = O.tensor_scale(w.numpy())
    return w, idx, nv().quantize(w.to(DEV)), st, O.quantize(w.numpy()[idx.numpy()], s_t=st)


@pytest.mark.parametrize("M", [1, 4, 8])
def test_draft_head_config(M):
    """248,320 x 5120 head, 32,768-id mask, 3 draft steps: the masked argmax
    is checked exactly against the oracle over all masked rows; the full-vocab
    argmax is checked by its value and by sampled rows."""
    m = nv()
    w, idx, qw, st, wq_masked = _head()
    idx_np = idx.numpy()
    for step in range(3):
        h = synth.draft_hidden(M, step)
        ids, logit = m.gather_gemv_argmax(h.to(DEV), qw, idx.to(DEV))
        # the oracle's masked head: rows idx in mask order
        logits, _ = O.gather_logits(h.float().numpy(), wq_masked, None)
        omax = logits.max(axis=1)
        margin = O.top2_margin(logits)
        for r in range(M):
            got = int(ids[r])
            assert got in set(idx_np.tolist())
            pos = int(np.nonzero(idx_np == got)[0][0])
            rms = np.sqrt(np.mean(logits[r] ** 2))
            if margin[r] > TOL:
                assert logits[r][pos] == omax[r]
            assert abs(float(logit[r]) - omax[r]) <= TOL * rms
    # full vocabulary: the winner's oracle logit matches and no sampled row beats it
    h = synth.draft_hidden(M, 0)
    ids, logit = m.gather_gemv_argmax(h.to(DEV), qw, None)
    rows = np.random.default_rng(5).choice(w.shape[0], 8192, replace=False)
    for r in range(M):
        cand = np.concatenate([rows, [int(ids[r])]])
        lg, _ = O.gather_logits(h.float().numpy()[r:r + 1], O.quantize(w.numpy()[cand], s_t=st), None)
        rms = np.sqrt(np.mean(lg ** 2))
        assert abs(lg[0, -1] - float(logit[r])) <= TOL * rms
        assert lg[0].max() <= float(logit[r]) + TOL * rms
