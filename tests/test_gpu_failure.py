"""Failure detection on the GPU without a fault: a bounded device wait that can
only run out (an mbarrier that nothing completes) must end by itself, record
the timeout in the device error word, and leave the context usable."""

import time

import pytest

import synth
from tests.gpu_util import assert_close, scan_on_gpu, to_f64, torch_mod

pytestmark = pytest.mark.gpu

ETIMEOUT = -5


def test_bounded_wait_times_out_and_reports():
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    assert mm.mamba_device_status() == 0          # nothing pending before
    t0 = time.perf_counter()
    mm.mamba_selftest_wait_timeout(20000)         # 20 ms limit
    assert mm.mamba_device_status() == ETIMEOUT   # the wait gave up and said so
    elapsed = time.perf_counter() - t0
    assert 0.015 < elapsed < 5.0, elapsed
    assert mm.mamba_device_status() == 0          # reading cleared the word
    # the context still runs the scan correctly afterwards
    import oracle
    inp = synth.scan_inputs(synth.TINY)
    y, fin = scan_on_gpu(inp)
    w = oracle.scan_inputs_f64(inp)
    yr, hr, _ = oracle.scan(w["u"], w["delta"], w["A"], w["B"], w["C"], dt_bias=w["dt_bias"],
                            D_skip=w["D_skip"], z=w["z"])
    assert_close(to_f64(y), yr, synth.F32)
    torch.cuda.synchronize()
