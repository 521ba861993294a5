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


@pytest.mark.parametrize("M", [1, 4, 12, 32])
@pytest.mark.parametrize("K", [512, 384])
def test_index_entries_outside_the_weight_are_skipped(M, K):
    """Rows gathered in place (M <= 8 whole-row streaming at K % 256 == 0,
    tile::gather4 above, the register-fed kernel at K = 384): entries outside
    [0, V) are never read nor reported, so the result equals the argmax over
    the valid entries; with no valid entry the id is -1."""
    m = nv()
    V = 3000
    w = synth.normal_f32((V, K), 0.02, seed=91)
    idx = synth.permutation_prefix(V, 700, seed=92).clone()
    bad = [3, 50, 400, 699]
    for pos, val in zip(bad, (-1, V, V + 7, -(2 ** 31))):
        idx[pos] = val
    good = np.array([i for i in range(len(idx)) if i not in bad])
    h = synth.normal_bf16((M, K), seed=93 + M)
    qw = m.quantize(w.to(DEV))
    ids, logit = m.gather_gemv_argmax(h.to(DEV), qw, idx.to(DEV))
    check_against_oracle(ids.cpu().numpy(), logit.cpu().numpy(), h.float().numpy(), O.quantize(w.numpy()),
                         idx.numpy()[good])
    none = torch.tensor([-1, V, -5, V + 1], dtype=torch.int32)
    ids0, logit0 = m.gather_gemv_argmax(h.to(DEV), qw, none.to(DEV))
    assert (ids0.cpu() == -1).all() and torch.isnan(logit0.cpu()).all()


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


def test_compact_head_bits_match_plain_decode():
    """Every fast path gated byte-identical to plain decode (Serving
    Qwen3.8-27B..., "Rules I learned the expensive way"), for the draft head
    on compact rows: at 32,768 rows x 5120 (256 row tiles, one GEMV pass
    without split-K) a token's winning logit rounded to bf16 is the plain
    GEMV's largest output and the winner's own output, and the token's id and
    logit bits are the same alone and inside batches of 5, 8, 9 and 32."""
    m = nv()
    V, N, K = 248320, 32768, 5120
    qw = m.quantize(synth.normal_f32((N, K), 0.02, seed=61).to(DEV))
    ids = synth.permutation_prefix(V, N, seed=62).to(DEV)
    pos = torch.full((V,), -1, dtype=torch.int64, device=DEV)
    pos[ids.long()] = torch.arange(N, device=DEV)
    tok = synth.normal_bf16((1, K), seed=63).to(DEV)
    seen = []
    for M in (1, 5, 8, 9, 32):
        x = synth.normal_bf16((M, K), seed=M + 300).to(DEV)
        x[M - 1] = tok[0]
        wid, logit = m.gemv_argmax(x, qw, ids)
        y = m.gemm_w4a16(x, qw).float()
        best = y.max(dim=1).values
        assert torch.equal(logit.to(torch.bfloat16).float(), best), M
        rows = pos[wid.long()]
        assert bool((rows >= 0).all())
        assert torch.equal(y[torch.arange(M, device=DEV), rows], best), M
        seen.append((int(wid[M - 1]), int(logit[M - 1:M].view(torch.int32)[0])))
    assert all(s == seen[0] for s in seen), seen


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


@functools.lru_cache(maxsize=1)
def _full_vocab_oracle():
    """The oracle's fp64 logits over all 248,320 head rows for the hidden
    states of the full-vocabulary checks: the 8-row hidden states of draft
    steps 0..2 (M = 1 and 4 are their first rows) and the 32-row verify batch.
    Returns {key: logits [rows][V]}."""
    from tests.head_oracle import full_head_logits
    _, _, _, st, _ = _head()
    hs = [synth.draft_hidden(8, s).float().numpy() for s in range(3)] + [synth.verify_hidden(32).float().numpy()]
    lg = full_head_logits(np.concatenate(hs), st)
    out = {("draft", s): lg[8 * s:8 * s + 8] for s in range(3)}
    out["verify"] = lg[24:56]
    return out


def check_full_vocab(ids, logit, logits):
    """The spec rule over every row of the head: the GPU id equals the
    oracle's (lowest id among equal maxima) wherever the oracle's top-2 margin
    exceeds the tolerance, and is one of the top two otherwise; its logit
    matches the oracle's maximum."""
    rows = np.arange(logits.shape[1])
    oid, omax = O.argmax_lowest_id(logits, rows)
    margin = O.top2_margin(logits)
    for r in range(len(ids)):
        rms = np.sqrt(np.mean(logits[r] ** 2))
        if margin[r] > TOL:
            assert int(ids[r]) == int(oid[r]), (r, margin[r])
        else:
            assert int(ids[r]) in set(np.argsort(logits[r])[-2:].tolist())
        assert abs(float(logit[r]) - omax[r]) <= TOL * rms


@pytest.mark.parametrize("M", [1, 4, 8])
def test_draft_head_config(M):
    """248,320 x 5120 head, 32,768-id mask, 3 draft steps: the masked argmax
    is checked exactly against the oracle over all masked rows, and the
    full-vocabulary argmax over all 248,320 rows."""
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
    # full vocabulary, every row of the head
    full = _full_vocab_oracle()
    for step in range(3):
        h = synth.draft_hidden(M, step)
        ids, logit = m.gather_gemv_argmax(h.to(DEV), qw, None)
        check_full_vocab(ids.cpu().numpy(), logit.cpu().numpy(), full[("draft", step)][:M])


def test_verify_head_full_vocab_m32():
    """The speculative verify shape: 32 rows (batch x (drafts + 1)) against
    the full 248,320-row head, through both entry points, checked over every
    row of the head."""
    m = nv()
    _, _, qw, _, _ = _head()
    h = synth.verify_hidden(32).to(DEV)
    full = _full_vocab_oracle()["verify"]
    ids, logit = m.gemv_argmax(h, qw, None)
    check_full_vocab(ids.cpu().numpy(), logit.cpu().numpy(), full)
    ids_g, logit_g = m.gather_gemv_argmax(h, qw, None)
    check_full_vocab(ids_g.cpu().numpy(), logit_g.cpu().numpy(), full)


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


def _drafts_from(target, V):
    """Drafts built from the oracle's own target tokens: sequence b gets its
    first b % (D + 1) drafts right and the next one wrong, so every accepted
    length 0..D occurs."""
    B, D1 = target.shape
    drafts = target[:, :D1 - 1].copy()
    for b in range(B):
        k = b % D1
        if k < D1 - 1:
            drafts[b, k] = (drafts[b, k] + 1) % V
    return drafts


def check_verify(tokens, n_acc, drafts, logits):
    B, D1 = tokens.shape
    V = logits.shape[1]
    oid, _ = O.argmax_lowest_id(logits, np.arange(V))
    target = oid.reshape(B, D1)
    n_ref = O.accept_greedy(target, drafts)
    margin = O.top2_margin(logits).reshape(B, D1)
    for b in range(B):
        # the count follows the returned tokens (greedy acceptance)
        assert int(n_acc[b]) == int(O.accept_greedy(tokens[b:b + 1], drafts[b:b + 1])[0])
        for i in range(D1):
            if margin[b, i] > TOL:
                assert int(tokens[b, i]) == int(target[b, i]), (b, i)
        if all(margin[b, i] > TOL for i in range(min(int(n_ref[b]), D1 - 1) + 1)):
            assert int(n_acc[b]) == int(n_ref[b]), b


@pytest.mark.parametrize("B,D", [(1, 0), (2, 3), (4, 7), (8, 3), (32, 0)])
def test_verify_accept_small_head(B, D):
    m = nv()
    V, K = 3000, 512
    w = synth.normal_f32((V, K), 0.02, seed=91)
    h = synth.normal_bf16((B * (D + 1), K), seed=92 + B)
    wq = O.quantize(w.numpy())
    ids, _, logits = O.gather_gemv_argmax(h.float().numpy(), wq, None)
    drafts = _drafts_from(ids.reshape(B, D + 1), V)
    tokens, n_acc = m.verify_accept(h.to(DEV), m.quantize(w.to(DEV)),
                                    torch.from_numpy(drafts.astype(np.int32)).to(DEV))
    check_verify(tokens.cpu().numpy(), n_acc.cpu().numpy(), drafts, logits)


def test_verify_accept_full_size():
    """Speculative verify at the 248,320 x 5120 head: 8 sequences x (3 drafts
    + 1) = 32 rows, every accepted length 0..3, against the oracle's logits
    over every row of the head."""
    m = nv()
    _, _, qw, _, _ = _head()
    logits = _full_vocab_oracle()["verify"]
    oid, _ = O.argmax_lowest_id(logits, np.arange(logits.shape[1]))
    drafts = _drafts_from(oid.reshape(8, 4), logits.shape[1])
    tokens, n_acc = m.verify_accept(synth.verify_hidden(32).to(DEV), qw,
                                    torch.from_numpy(drafts.astype(np.int32)).to(DEV))
    check_verify(tokens.cpu().numpy(), n_acc.cpu().numpy(), drafts, logits)
