"""W4A16 decode GEMV / skinny GEMM parity against the fp64 oracle."""
import functools

import numpy as np
import pytest
import torch

import oracle as O
import synth
from tests.gpu_common import DEV, np_f64, nv

pytestmark = pytest.mark.gpu
TOL = 1e-2


def run(w_f32, x_bf16):
    m = nv()
    qw = m.quantize(w_f32.to(DEV))
    y = m.gemm_w4a16(x_bf16.to(DEV), qw)
    return np_f64(y), O.gemm_w4a16(x_bf16.float().numpy(), O.quantize(w_f32.numpy()))


def test_tiny_config():
    w, x = synth.tiny_w4a16(seed=0)
    y, ref = run(w, x)
    assert O.rel_fro(y, ref) <= TOL
    assert np.max(np.abs(y - ref)) / np.max(np.abs(ref)) <= TOL


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 9, 17, 32, 33, 70])
@pytest.mark.parametrize("N,K", [(512, 256), (200, 384), (136, 1280), (200, 512)])
def test_shapes(M, N, K):
    w = synth.normal_f32((N, K), 0.02, seed=N + K)
    x = synth.normal_bf16((M, K), seed=M)
    y, ref = run(w, x)
    assert O.rel_fro(y, ref) <= TOL, (M, N, K)


def test_exact_special_case_is_bit_exact():
    """Power-of-two scales, s_t = 1, activations in {-8..8}/8: every partial
    sum is exact in fp32, so the bf16 output must equal the rounded fp64 sum."""
    m = nv()
    rng = np.random.default_rng(1)
    N, K, M = 512, 256, 4
    codes = rng.integers(0, 16, (N, K)).astype(np.uint8)
    exps = rng.integers(-3, 4, (N, K // 16))
    scales = (((exps + 7) << 3)).astype(np.uint8)
    qref = O.QTensor(O.pack_codes(codes), scales, 1.0)
    x = torch.from_numpy(rng.integers(-8, 9, (M, K)).astype(np.float32) / 8).to(torch.bfloat16)
    qw = m.QTensor(torch.from_numpy(qref.codes).to(DEV), torch.from_numpy(qref.scales).to(DEV),
                   torch.ones(1, device=DEV), N, K)
    y = m.gemm_w4a16(x.to(DEV), qw).float().cpu().numpy()
    ref = O.bf16_round(O.gemm_w4a16(x.float().numpy(), qref))
    assert np.array_equal(y, ref)


def test_large_activation_range():
    """Activations far outside f16 range (and tiny ones) still match."""
    w = synth.normal_f32((256, 512), 0.02, seed=3)
    x = (synth.normal_f32((4, 512), 1.0, seed=4) * torch.tensor([[1e6], [1e-6], [3e30], [1.0]])).to(torch.bfloat16)
    y, ref = run(w, x)
    for r in range(4):
        assert O.rel_fro(y[r], ref[r]) <= TOL


@functools.lru_cache(maxsize=1)
def _decode_weight(which):
    """(fp32 weight, its GPU quantisation, the oracle's tensor scale)."""
    w = synth.decode_weight(which)
    return w, nv().quantize(w.to(DEV)), O.tensor_scale(w.numpy())


@pytest.mark.parametrize("which", ["gate_up", "down"])
@pytest.mark.parametrize("M", [1, 4, 8, 32])
def test_decode_config_sampled_rows(which, M):
    """27B decode linears at full size, the bench's launch; output columns
    sampled and recomputed by the oracle one by one."""
    m = nv()
    w, qw, st = _decode_weight(which)
    N, K = w.shape
    x = synth.decode_activation(M, K)
    y = np_f64(m.gemm_w4a16(x.to(DEV), qw))
    cols = np.sort(np.random.default_rng(M).choice(N, 384, replace=False))
    ref = O.gemm_w4a16(x.float().numpy(), O.quantize(w.numpy()[cols], s_t=st))
    assert O.rel_fro(y[:, cols], ref) <= TOL


def test_split_k_is_deterministic_and_matches_unsplit_shape():
    """N small enough that the K range is split across CTAs: two calls give
    identical bits, and the result matches the oracle."""
    m = nv()
    w = synth.normal_f32((256, 8192), 0.02, seed=61)
    x = synth.normal_bf16((5, 8192), seed=62)
    qw = m.quantize(w.to(DEV))
    a = m.gemm_w4a16(x.to(DEV), qw)
    b = m.gemm_w4a16(x.to(DEV), qw)
    assert torch.equal(a, b)
    ref = O.gemm_w4a16(x.float().numpy(), O.quantize(w.numpy()))
    assert O.rel_fro(np_f64(a), ref) <= TOL


@pytest.mark.parametrize("N,K", [(256, 2048), (128, 8192)])
def test_activation_magnitude_changes_along_k(N, K):
    """Tokens whose magnitude jumps between 256-element stretches of K: the
    in-kernel conversion raises its power-of-two shift mid-row and rescales
    the accumulators (the second shape also splits K across CTAs)."""
    w = synth.normal_f32((N, K), 0.02, seed=71)
    x = synth.normal_f32((7, K), 1.0, seed=72)
    nb = K // 256
    b = torch.arange(nb, dtype=torch.float32)
    blocks = torch.stack([
        2.0 ** (4 * b),                                  # growing
        2.0 ** (-4 * b),                                 # shrinking
        torch.where(b < nb // 2, 0.0, 1.0),              # zeros, then values
        torch.where(b == nb - 1, 3e30, 1.0),             # one huge stretch at the end
        torch.zeros(nb),                                 # all zero
        torch.where(b % 2 == 0, 1e-20, 1e20),            # alternating tiny / huge
        torch.ones(nb),
    ])
    x = (x * blocks.repeat_interleave(256, dim=1)).to(torch.bfloat16)
    y, ref = run(w, x)
    assert np.all(y[4] == 0.0)
    for r in (0, 1, 2, 3, 5, 6):
        assert O.rel_fro(y[r], ref[r]) <= TOL, r


@pytest.mark.parametrize("N,K", [(1000, 2048), (5120, 17408), (300, 384), (34816, 5120)])
def test_token_bits_do_not_depend_on_batch(N, K):
    """Every fast path gated byte-identical to plain decode (Serving
    Qwen3.8-27B..., "Rules I learned the expensive way"): one token's output
    row is bit for bit the same whether it runs alone or inside batches of 8,
    17, 32 (the shape buckets of decode), 33 or 70 tokens (several token
    chunks), at a split-K shape (17408 -> 5120), a single-pass one (5120 ->
    34816) and the register-fed kernel (K = 384)."""
    m = nv()
    qw = m.quantize(synth.normal_f32((N, K), 0.02, seed=N + 3 * K).to(DEV))
    tok = synth.normal_bf16((1, K), seed=K + 1).to(DEV)
    rows = []
    for M in (1, 8, 17, 32, 33, 70):
        x = synth.normal_bf16((M, K), seed=M + 100).to(DEV)
        pos = M - 1                        # the last row: another token chunk once M > 32
        x[pos] = tok[0]
        rows.append(m.gemm_w4a16(x, qw)[pos].clone())
    for M, r in zip((8, 17, 32, 33, 70), rows[1:]):
        assert torch.equal(r.view(torch.int16), rows[0].view(torch.int16)), M


def silu_mul_ref(x_bf16, wq_gate, wq_up):
    """Oracle: h = bf16(silu(g) * u) from fp64 g, u (reading R7 on a dense layer)."""
    x = x_bf16.float().numpy()
    return O.bf16_round(O.silu(O.gemm_w4a16(x, wq_gate)) * O.gemm_w4a16(x, wq_up))


@pytest.mark.parametrize("M", [1, 5, 32, 40])
@pytest.mark.parametrize("I,K", [(128, 4096), (256, 256), (192, 1024)])
def test_silu_mul_fused_gate_up(M, I, K):
    """(128, 4096) splits K across CTAs; (256, 256) does not; M = 40 spans two token chunks."""
    m = nv()
    w = synth.normal_f32((2 * I, K), 0.02, seed=I + K)
    x = synth.normal_bf16((M, K), seed=M + 7)
    h = np_f64(m.gemm_w4a16_silu_mul(x.to(DEV), m.quantize(w.to(DEV))))
    st = O.tensor_scale(w.numpy())
    ref = silu_mul_ref(x, O.quantize(w.numpy()[:I], s_t=st), O.quantize(w.numpy()[I:], s_t=st))
    assert h.shape == (M, I)
    assert O.rel_fro(h, ref) <= TOL


@pytest.mark.parametrize("M", [1, 8, 32])
def test_silu_mul_27b_gate_up_sampled(M):
    """The 27B gate/up (5120 -> 2 x 17408) with SiLU * mul fused: 256 sampled
    intermediate columns against the oracle (gate row i and up row I + i,
    quantised with the whole tensor's scale)."""
    m = nv()
    wt, qw, st = _decode_weight("gate_up")
    w = wt.numpy()
    I = w.shape[0] // 2
    x = synth.decode_activation(M, w.shape[1])
    h = np_f64(m.gemm_w4a16_silu_mul(x.to(DEV), qw))
    cols = np.sort(np.random.default_rng(M).choice(I, 256, replace=False))
    ref = silu_mul_ref(x, O.quantize(w[cols], s_t=st), O.quantize(w[I + cols], s_t=st))
    assert O.rel_fro(h[:, cols], ref) <= TOL


def test_silu_mul_rows_do_not_depend_on_batch():
    m = nv()
    I, K = 256, 4096
    qw = m.quantize(synth.normal_f32((2 * I, K), 0.02, seed=77).to(DEV))
    tok = synth.normal_bf16((1, K), seed=78).to(DEV)
    rows = []
    for M in (1, 9, 32, 33):
        x = synth.normal_bf16((M, K), seed=M + 200).to(DEV)
        x[M - 1] = tok[0]
        rows.append(m.gemm_w4a16_silu_mul(x, qw)[M - 1].clone())
    for r in rows[1:]:
        assert torch.equal(r.view(torch.int16), rows[0].view(torch.int16))
