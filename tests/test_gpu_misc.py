"""Failure detection on the device: a bounded wait that runs out reports an
error instead of hanging, and the context stays usable afterwards."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from tests.gpu_common import DEV, np_u8, nv

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    m = nv()
    assert m.read_device_status() == 0
    m.selftest_bounded_wait(2_000_000)          # 2 ms, nothing ever arrives
    assert m.read_device_status() == -6
    assert m.read_device_status() == 0          # reading clears it
    x = synth.normal_f32((8, 64), 1.0, seed=1)
    q = m.quantize(x.to(DEV))
    assert np.array_equal(np_u8(q.codes), O.quantize(x.numpy()).codes)


def test_status_clean_after_gemm():
    m = nv()
    a = synth.student_t_bf16((256, 256), 4, seed=2)
    w = synth.normal_f32((256, 256), 0.02, seed=3)
    m.gemm_w4a4(m.quantize(a.to(DEV), scale_layout=1), m.prepack_scales(m.quantize(w.to(DEV))))
    assert m.read_device_status() == 0


def test_errors_are_reported_not_raised_on_device():
    m = nv()
    x = torch.zeros(4, 40, device=DEV)
    with pytest.raises(RuntimeError, match="unsupported shape"):
        m.quantize(x)
