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


def test_fp4_mma_rate_probe_runs_and_reports_ok():
    """The FP4 tensor-pipe ceiling probe finishes (its bounded wait does not
    give up) and its rate is a plausible fraction of the nominal dense FP4
    figure: above 1 PFLOP/s, below 20."""
    m = nv()
    m.read_device_status()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    m.probe_fp4_mma_rate(100)   # warm-up
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    m.probe_fp4_mma_rate(20000)
    b.record()
    torch.cuda.synchronize()
    assert m.read_device_status() == m.OK
    pflops = sms * 20000 * 2.0 * 128 * 256 * 64 / (a.elapsed_time(b) * 1e-3) / 1e15
    assert 1.0 < pflops < 20.0, pflops
