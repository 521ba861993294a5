"""Quantiser parity: codes, block scales and tensor scale bit-exact against
the oracle, for every layout, dtype and scale mode."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from tests.gpu_common import DEV, np_u8, nv, unpack_mma_scales
from tests.test_oracle import load_blocks

pytestmark = pytest.mark.gpu


def check(qt_gpu, qt_ref, layout):
    assert np.array_equal(np_u8(qt_gpu.codes), qt_ref.codes)
    if layout == 0:
        got = np_u8(qt_gpu.scales)
    else:
        got = unpack_mma_scales(np_u8(qt_gpu.scales), qt_ref.codes.shape[0], qt_ref.codes.shape[1] * 2)
    assert np.array_equal(got, qt_ref.scales)
    assert np.float32(qt_gpu.s_t.item()) == qt_ref.s_t


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_golden_blocks(dtype):
    m = nv()
    for blk in load_blocks():
        x = torch.tensor([blk["x"]], dtype=torch.float32).to(dtype)
        q = m.quantize(x.to(DEV), s_t=torch.tensor([blk["s_t"]]))
        assert int(np_u8(q.scales)[0, 0]) == blk["scale"], blk["name"]
        assert list(np_u8(q.codes)[0]) == blk["packed"], blk["name"]


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("case", ["weights_f32", "act_bf16", "student_t", "ragged", "k16", "tiny_values"])
def test_random_tensors_bit_exact(case, layout):
    m = nv()
    if case == "weights_f32":
        x = synth.normal_f32((512, 256), 0.02, seed=0)
    elif case == "act_bf16":
        x = synth.normal_bf16((64, 5120), seed=2)
    elif case == "student_t":
        x = synth.student_t_bf16((300, 1024), 4, seed=3)
    elif case == "ragged":
        x = synth.normal_f32((131, 208), 1.0, seed=11)
    elif case == "k16":
        x = synth.normal_bf16((7, 16), seed=12)
    else:
        # magnitudes spanning E4M3 subnormal block scales
        x = synth.normal_f32((96, 512), 1.0, seed=13) * torch.logspace(-6, 1, 512)
    q = m.quantize(x.to(DEV), scale_layout=layout)
    check(q, O.quantize(x.float().numpy()), layout)


def test_given_scale_and_saturation():
    m = nv()
    x = synth.normal_f32((64, 128), 3.0, seed=14)
    q = m.quantize(x.to(DEV), s_t=torch.tensor([0.0005]))   # far too small: scales and codes saturate
    check(q, O.quantize(x.numpy(), s_t=np.float32(0.0005)), 0)


def test_zero_tensor_and_empty():
    m = nv()
    z = torch.zeros(4, 64)
    z[1, 3] = -0.0
    q = m.quantize(z.to(DEV))
    assert q.s_t.item() == 1.0
    assert np_u8(q.codes).max() == 0 and np_u8(q.scales).max() == 0
    e = m.quantize(torch.zeros(0, 64, device=DEV))
    assert e.s_t.item() == 1.0


def test_prepack_matches_direct_mma_quantise():
    m = nv()
    x = synth.normal_f32((300, 320), 0.02, seed=15)
    a = m.prepack_scales(m.quantize(x.to(DEV)))
    b = m.quantize(x.to(DEV), scale_layout=m.SCALES_MMA)
    assert torch.equal(a.scales, b.scales)


def test_full_size_weight_sampled_rows():
    """27B gate/up weight [34816][5120]: quantised on the GPU in one call; 256
    sampled rows re-quantised by the oracle with the oracle's own full-tensor
    scale."""
    m = nv()
    w = synth.decode_weight("gate_up")
    q = m.quantize(w.to(DEV))
    st = O.tensor_scale(w.numpy())
    assert np.float32(q.s_t.item()) == st
    rows = np.sort(np.random.default_rng(0).choice(w.shape[0], 256, replace=False))
    ref = O.quantize(w.numpy()[rows], s_t=st)
    assert np.array_equal(np_u8(q.codes[rows]), ref.codes)
    assert np.array_equal(np_u8(q.scales[rows]), ref.scales)


def test_full_size_prefill_activations_mma_layout():
    """8192 x 5120 Student-t activations straight into the MMA layout, every
    element checked."""
    m = nv()
    a = synth.prefill_inputs(M=8192)[0]
    q = m.quantize(a.to(DEV), scale_layout=m.SCALES_MMA)
    check(q, O.quantize(a.float().numpy()), 1)


def test_values_next_to_rounding_midpoints():
    """Element quotients a few ulps either side of every e2m1 rounding
    midpoint (and exactly on it), for many block scales: the code decision
    there must equal the one the IEEE-divided quotient gives."""
    m = nv()
    rng = np.random.default_rng(21)
    rows, blocks = 256, 32
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float64)
    # block scales: E4M3 normals 2^-6 .. 448 (mantissas 1 + j/8)
    exps = rng.integers(-6, 9, size=(rows, blocks))
    mans = 1.0 + rng.integers(0, 8, size=(rows, blocks)) / 8.0
    den = np.minimum(mans * np.exp2(exps), 448.0)
    x = np.empty((rows, blocks, 16), dtype=np.float32)
    x[:, :, 0] = (6.0 * den).astype(np.float32)          # the block amax: scale == den exactly (s_t = 1)
    mid = rng.choice(mids, size=(rows, blocks, 15))
    k = rng.integers(-4, 5, size=(rows, blocks, 15))
    q = (mid * (1.0 + k * 2.0 ** -23)).astype(np.float32)
    x[:, :, 1:] = (q.astype(np.float64) * den[:, :, None]).astype(np.float32)
    x *= np.where(rng.random(x.shape) < 0.5, -1.0, 1.0).astype(np.float32)
    x[:, :, 0] = np.abs(x[:, :, 0])
    x = x.reshape(rows, blocks * 16)
    for layout in (0, 1):
        qg = m.quantize(torch.from_numpy(x).to(DEV), s_t=torch.tensor([1.0]), scale_layout=layout)
        check(qg, O.quantize(x, s_t=np.float32(1.0)), layout)
