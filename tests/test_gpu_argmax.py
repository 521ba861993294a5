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


@functools.lru_cache(maxsize=1)
def _compact():
    _, idx, qw, _, _ = _head()
    return nv().gather_rows(qw, idx.to(DEV))


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
        # the same head as a compact prepacked copy of the masked rows
        ids_c, logit_c = m.gemv_argmax(h.to(DEV), _compact(), idx.to(DEV))
        for r in range(M):
            for got, lg in ((int(ids[r]), float(logit[r])), (int(ids_c[r]), float(logit_c[r]))):
                assert got in set(idx_np.tolist())
                pos = int(np.nonzero(idx_np == got)[0][0])
                rms = np.sqrt(np.mean(logits[r] ** 2))
                if margin[r] > TOL:
                    assert logits[r][pos] == omax[r]
                assert abs(lg - omax[r]) <= TOL * rms
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


def test_gather_rows_matches_the_oracles_rows_byte_for_byte():
    m = nv()
    V, K = 2000, 512
    w = synth.normal_f32((V, K), 0.02, seed=51)
    idx = synth.permutation_prefix(V, 333, seed=52)
    sub = m.gather_rows(m.quantize(w.to(DEV)), idx.to(DEV))
    ref = O.quantize(w.numpy()[idx.numpy()], s_t=O.tensor_scale(w.numpy()))
    assert np.array_equal(sub.codes.cpu().numpy(), ref.codes)
    assert np.array_equal(sub.scales.cpu().numpy().reshape(ref.scales.shape), ref.scales)


@pytest.mark.parametrize("M", [1, 5, 8, 13, 32])
def test_gemv_argmax_on_compact_rows_equals_masked_head(M):
    """The compact copy of the masked rows with the mask as id map gives the
    masked head's answer (checked against the oracle as well)."""
    m = nv()
    V, K = 4000, 512
    w = synth.normal_f32((V, K), 0.02, seed=61)
    idx = synth.permutation_prefix(V, 1000, seed=62)
    h = synth.normal_bf16((M, K), seed=63 + M)
    qw = m.quantize(w.to(DEV))
    ids, logit = m.gemv_argmax(h.to(DEV), m.gather_rows(qw, idx.to(DEV)), idx.to(DEV))
    check_against_oracle(ids.cpu().numpy(), logit.cpu().numpy(), h.float().numpy(), O.quantize(w.numpy()),
                         idx.numpy())
    ids_g, _ = m.gather_gemv_argmax(h.to(DEV), qw, idx.to(DEV))
    _, _, logits = O.gather_gemv_argmax(h.float().numpy(), O.quantize(w.numpy()), idx.numpy())
    margin = O.top2_margin(logits)
    for r in range(M):
        if margin[r] > TOL:
            assert int(ids[r]) == int(ids_g[r])


def test_gather_rows_out_of_range_index_is_reported():
    m = nv()
    qw = m.quantize(synth.normal_f32((64, 256), 0.02, seed=71).to(DEV))
    idx = torch.tensor([3, 64, 5], dtype=torch.int32, device=DEV)
    m.read_device_status()   # clear
    sub = m.gather_rows(qw, idx)
    assert m.read_device_status() == m.ERR_INVALID_ARG
    assert int(sub.codes[1].abs().sum()) == 0 and torch.equal(sub.codes[0], qw.codes[3])
