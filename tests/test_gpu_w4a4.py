"""W4A4 prefill GEMM on the block-scaled FP4 tensor cores, against the
fp64 oracle on the oracle's own quantisation of the same inputs."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from tests.gpu_common import DEV, np_f64, nv

pytestmark = pytest.mark.gpu
TOL = 1e-2


def gpu_gemm(a_bf16, w_f32, a_layout=1, w_layout=1):
    m = nv()
    qa = m.quantize(a_bf16.to(DEV), scale_layout=a_layout)
    qw = m.quantize(w_f32.to(DEV))
    if w_layout == 1:
        qw = m.prepack_scales(qw)
    return np_f64(m.gemm_w4a4(qa, qw))


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 256, 512), (200, 136, 320), (1, 8, 64),
                                   (384, 512, 1024), (130, 264, 576), (640, 256, 256), (1024, 520, 768)])
@pytest.mark.parametrize("layouts", [(1, 1), (0, 0)])
def test_shapes(M, N, K, layouts):
    a = synth.student_t_bf16((M, K), 4, seed=M)
    w = synth.normal_f32((N, K), 0.02, seed=N)
    y = gpu_gemm(a, w, *layouts)
    ref = O.gemm_w4a4(O.quantize(a.float().numpy()), O.quantize(w.numpy()))
    assert O.rel_fro(y, ref) <= TOL, (M, N, K, O.rel_fro(y, ref))


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 256, 512), (384, 264, 320), (640, 520, 1024),
                                   (4096, 4096, 128)])
def test_exact_special_case_is_bit_exact(M, N, K):
    """Unit scales and s_t = 1 on both sides: products of e2m1 codes are exact
    and every partial sum is a small multiple of 1/4, so the output is exact.
    M > 128 runs the CTA-pair kernel (odd m-tile counts, ragged N and K; the
    largest shape gives each CTA pair several tiles in turn)."""
    m = nv()
    rng = np.random.default_rng(2)
    ca = rng.integers(0, 16, (M, K)).astype(np.uint8)
    cw = rng.integers(0, 16, (N, K)).astype(np.uint8)
    one = np.full((M, K // 16), 0x38, np.uint8)
    qa_ref = O.QTensor(O.pack_codes(ca), one, 1.0)
    qw_ref = O.QTensor(O.pack_codes(cw), np.full((N, K // 16), 0x38, np.uint8), 1.0)
    dev = lambda a: torch.from_numpy(a).to(DEV)
    qa = m.QTensor(dev(qa_ref.codes), dev(qa_ref.scales), torch.ones(1, device=DEV), M, K)
    qw = m.QTensor(dev(qw_ref.codes), dev(qw_ref.scales), torch.ones(1, device=DEV), N, K)
    y = np_f64(m.gemm_w4a4(qa, qw))
    assert np.array_equal(y, O.bf16_round(O.gemm_w4a4(qa_ref, qw_ref)))


def test_reduces_to_w4a16_on_decoded_activations():
    m = nv()
    a = synth.student_t_bf16((64, 512), 4, seed=5)
    w = synth.normal_f32((256, 512), 0.02, seed=6)
    y4 = gpu_gemm(a, w)
    aq = O.quantize(a.float().numpy())
    ref = O.gemm_w4a16(O.decode(aq), O.quantize(w.numpy()))
    assert O.rel_fro(y4, ref) <= TOL


def test_prefill_config_sampled():
    """M=8192, K=5120, N=34816 at full size; 128 rows x 1024 columns of the
    output recomputed by the oracle."""
    m = nv()
    a, w = synth.prefill_inputs()
    qa = m.quantize(a.to(DEV), scale_layout=m.SCALES_MMA)
    qw = m.prepack_scales(m.quantize(w.to(DEV)))
    y = m.gemm_w4a4(qa, qw)
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(a.shape[0], 128, replace=False))
    cols = np.sort(rng.choice(w.shape[0], 1024, replace=False))
    ys = np_f64(y[torch.from_numpy(rows).to(DEV)][:, torch.from_numpy(cols).to(DEV)])
    a_np, w_np = a.float().numpy(), w.numpy()
    ra = O.quantize(a_np[rows], s_t=O.tensor_scale(a_np))
    rw = O.quantize(w_np[cols], s_t=O.tensor_scale(w_np))
    assert O.rel_fro(ys, O.gemm_w4a4(ra, rw)) <= TOL


def _exact_operands(M, N, K, seed=2):
    """Codes of both operands random, unit scales, s_t = 1: every product is
    exact and every partial sum a small multiple of 1/4, exact in fp32."""
    m = nv()
    rng = np.random.default_rng(seed)
    ca = rng.integers(0, 16, (M, K)).astype(np.uint8)
    cw = rng.integers(0, 16, (N, K)).astype(np.uint8)
    qa_ref = O.QTensor(O.pack_codes(ca), np.full((M, K // 16), 0x38, np.uint8), 1.0)
    qw_ref = O.QTensor(O.pack_codes(cw), np.full((N, K // 16), 0x38, np.uint8), 1.0)
    dev = lambda a: torch.from_numpy(a).to(DEV)
    qa = m.QTensor(dev(qa_ref.codes), dev(qa_ref.scales), torch.ones(1, device=DEV), M, K)
    qw = m.QTensor(dev(qw_ref.codes), dev(qw_ref.scales), torch.ones(1, device=DEV), N, K)
    return qa, qw, qa_ref, qw_ref


def mma_scale_buffer(scales, rows, K):
    """The whole MMA-layout buffer (padding zero) for row-major scales, from
    the layout's definition in include/nvfp4.h."""
    kc = K // 16
    rp, cp = (rows + 127) // 128 * 128, (kc + 3) // 4 * 4
    buf = np.zeros(rp * cp, np.uint8)
    r = np.arange(rows)[:, None]
    c = np.arange(kc)[None, :]
    off = ((r // 128) * (cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4
    buf[off] = scales
    return buf


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 256, 512), (384, 320, 320), (200, 192, 128),
                                   (640, 576, 1024), (1, 64, 64)])
def test_quant_epilogue_exact_case_is_bit_exact(M, N, K):
    """The W4A4 output handed on as NVFP4: where the GEMM is exact its bf16
    output equals the oracle's, so the codes and MMA-layout scales (padding
    included) must equal the oracle's quantisation of it bit for bit - with a
    given tensor scale (fused epilogue) and with the dynamic one (GEMM + amax,
    then the quantiser). (128, ...) runs the single-CTA kernel, the rest the
    pair kernel with odd m-tile counts and ragged N."""
    m = nv()
    qa, qw, qa_ref, qw_ref = _exact_operands(M, N, K)
    yb = O.bf16_round(O.gemm_w4a4(qa_ref, qw_ref)).astype(np.float32)
    st_given = np.float32(0.0371)
    ref = O.gemm_w4a4_nvfp4(qa_ref, qw_ref, s_t=st_given)
    q = m.gemm_w4a4_quant(qa, qw, s_t=torch.tensor([float(st_given)]))
    assert np.array_equal(q.codes.cpu().numpy(), ref.codes)
    assert np.array_equal(q.scales.cpu().numpy(), mma_scale_buffer(ref.scales, M, N))
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    qd = m.gemm_w4a4_quant(qa, qw, y=y)
    refd = O.gemm_w4a4_nvfp4(qa_ref, qw_ref)
    assert np.float32(qd.s_t.item()) == refd.s_t
    assert np.array_equal(qd.codes.cpu().numpy(), refd.codes)
    assert np.array_equal(qd.scales.cpu().numpy(), mma_scale_buffer(refd.scales, M, N))
    assert np.array_equal(y.float().cpu().numpy(), yb)


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (96, 256, 512), (640, 320, 768)])
def test_quant_epilogue_general_inputs(M, N, K):
    """Student-t activations, N(0, 0.02) weights: the NVFP4 output decodes to
    the oracle's quantisation of the oracle's bf16 output within tolerance,
    and almost every code matches exactly (the two bf16 outputs differ only
    where the fp32 and fp64 sums round to different bf16 values)."""
    m = nv()
    a = synth.student_t_bf16((M, K), 4, seed=M + 1)
    w = synth.normal_f32((N, K), 0.02, seed=N + 1)
    qa = m.quantize(a.to(DEV), scale_layout=m.SCALES_MMA)
    qw = m.prepack_scales(m.quantize(w.to(DEV)))
    oa, ow = O.quantize(a.float().numpy()), O.quantize(w.numpy())
    yb = O.bf16_round(O.gemm_w4a4(oa, ow)).astype(np.float32)
    st = np.float32(O.tensor_scale(yb) * np.float32(1.25))
    ref = O.gemm_w4a4_nvfp4(oa, ow, s_t=st)
    q = m.gemm_w4a4_quant(qa, qw, s_t=torch.tensor([float(st)]))
    from tests.gpu_common import unpack_mma_scales
    got = O.QTensor(q.codes.cpu().numpy(), unpack_mma_scales(q.scales.cpu().numpy(), M, N), st)
    assert O.rel_fro(O.decode(got), O.decode(ref)) <= TOL
    assert np.mean(got.codes != ref.codes) < 0.02
    qd = m.gemm_w4a4_quant(qa, qw)
    assert abs(float(qd.s_t.item()) / float(O.tensor_scale(yb)) - 1.0) <= TOL
