"""Run by tests/test_gpu_debug_build.py in a fresh process with
MAMBA_SCAN_LIBRARY=debug: drives the library built with -DMAMBA_DEBUG
(index checks on every global access) through the odd scan shapes, the
generation step, the convolution, the backward pass and the training pair,
checks each against the fp64 oracle, and checks that no index check failed.
Also runs the index-check self-test, which must be reported as
MAMBA_ERR_BOUNDS with its source line."""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402
import selective_state_space_135_b300 as mm  # noqa: E402
from tests.gpu_util import assert_close, f32_dev, scan_on_gpu, to_dev, to_f64  # noqa: E402
from tests.test_gpu_scan import ODD  # noqa: E402

BOUNDS = -11


def main():
    assert os.path.basename(mm.lib_path()) == "libmamba_scan_debug.so", mm.lib_path()
    is_debug, line = mm.mamba_debug_build()
    assert is_debug and line == 0
    # scans: every odd shape (tensor-map and element-wise paths, ragged tails)
    for dtype, batch, dim, n, l in ODD:
        shp = synth.ScanShape("odd", batch, dim, n, l, dtype=dtype, seed=77 + l + dim)
        inp = synth.scan_inputs(shp)
        y, fin = scan_on_gpu(inp)
        assert mm.mamba_device_status() == 0, (shp, mm.mamba_debug_build())
        w = oracle.scan_inputs_f64(inp)
        yr, hr, _ = oracle.scan(w["u"], w["delta"], w["A"], w["B"], w["C"], dt_bias=w["dt_bias"],
                                D_skip=w["D_skip"], z=w["z"])
        assert_close(to_f64(y), yr, dtype)
        assert_close(to_f64(fin), hr, dtype, "final_state")
    # a chunked plan (summary, carry, main passes) and the extended modes
    shp = synth.ScanShape("chunked", 2, 100, 16, 520, seed=5)
    inp = synth.scan_inputs(shp)
    mm.mamba_scan_set_tuning(0, 0, 3)
    try:
        y, fin = scan_on_gpu(inp)
    finally:
        mm.mamba_scan_set_tuning(0, 0, 0)
    assert mm.mamba_device_status() == 0
    h0 = f32_dev(np.full((2, 100, 16), 0.25, np.float32))
    lens = torch.tensor([520, 17], dtype=torch.int32, device="cuda")
    mm.mamba_scan_fwd_ex(to_dev(inp["u"], shp.dtype), to_dev(inp["delta"], shp.dtype),
                         f32_dev(inp["dt_bias"]), f32_dev(inp["A"]), to_dev(inp["B"], shp.dtype),
                         to_dev(inp["C"], shp.dtype), f32_dev(inp["D_skip"]),
                         to_dev(inp["z"], shp.dtype), zoh=True, initial_state=h0, seqlens=lens)
    assert mm.mamba_device_status() == 0
    # generation steps: the dstate-16 vector kernel and the generic one
    for n, dtype in ((16, synth.BF16), (13, synth.F32)):
        dshp = synth.DecodeShape("step", 3, 70, n, 2, dtype=dtype, seed=8)
        par = synth.decode_params(dshp)
        state = torch.zeros((3, 70, n), device="cuda")
        si = synth.decode_step_inputs(dshp, 0)
        y = mm.mamba_state_update(state, to_dev(si["x"], dtype), to_dev(si["delta"], dtype),
                                  f32_dev(par["dt_bias"]), f32_dev(par["A"]), to_dev(si["B"], dtype),
                                  to_dev(si["C"], dtype), f32_dev(par["D_skip"]),
                                  to_dev(si["z"], dtype))
        assert mm.mamba_device_status() == 0
        yr = oracle.state_update(np.zeros((3, 70, n)), synth.widen(si["x"], dtype),
                                 synth.widen(si["delta"], dtype), par["A"],
                                 synth.widen(si["B"], dtype), synth.widen(si["C"], dtype),
                                 dt_bias=par["dt_bias"], D_skip=par["D_skip"],
                                 z=synth.widen(si["z"], dtype))
        assert_close(to_f64(y), yr, dtype)
    # the convolution and its step, ragged and aligned rows
    g = np.random.default_rng(21)
    for l in (37, 64):
        xb = synth.store(g.standard_normal((2, 24, l)).astype(np.float32), synth.BF16)
        x = to_dev(xb, synth.BF16)
        wt = f32_dev(g.standard_normal((24, 4)).astype(np.float32))
        st = torch.zeros((2, 24, 3), dtype=torch.bfloat16, device="cuda")
        fin = torch.empty_like(st)
        out = mm.mamba_conv1d_fwd(x, wt, None, conv_state=st, silu=True, final_conv_state=fin)
        mm.mamba_conv1d_update(fin, x[:, :, 0].contiguous(), wt, None, silu=True)
        assert mm.mamba_device_status() == 0
        ref = oracle.conv1d(synth.widen(xb, synth.BF16), wt.cpu().numpy().astype(np.float64),
                            silu=True)[0]
        assert_close(to_f64(out), ref, synth.BF16)
    # the backward pass (ragged tile, partial channel group, dstate 5 and 16,
    # 97 channel groups for the four-part reduction) and the training pair
    for dtype, batch, dim, n, l in ((synth.F32, 2, 33, 5, 70), (synth.BF16, 2, 70, 16, 200),
                                    (synth.BF16, 1, 3104, 16, 40)):
        shp = synth.ScanShape("debug bwd", batch, dim, n, l, dtype=dtype, seed=23)
        inp = synth.scan_inputs(shp)
        gg = np.random.default_rng(24)
        dyh = synth.store(gg.standard_normal((batch, dim, l)).astype(np.float32), dtype)
        h0 = (0.5 * gg.standard_normal((batch, dim, n))).astype(np.float32)
        dfin = gg.standard_normal((batch, dim, n)).astype(np.float32)
        args = (to_dev(inp["u"], dtype), to_dev(inp["delta"], dtype), f32_dev(inp["dt_bias"]),
                f32_dev(inp["A"]), to_dev(inp["B"], dtype), to_dev(inp["C"], dtype),
                f32_dev(inp["D_skip"]), to_dev(inp["z"], dtype))
        dy = to_dev(dyh, dtype)
        g1 = mm.mamba_scan_bwd(*args, dy, initial_state=f32_dev(h0), d_final_state=f32_dev(dfin),
                               want_initial_state_grad=True)
        _, ck = mm.mamba_scan_fwd_train(*args, initial_state=f32_dev(h0))
        g2 = mm.mamba_scan_bwd_ckpt(*args, dy, ck, d_final_state=f32_dev(dfin),
                                    want_initial_state_grad=True)
        torch.cuda.synchronize()
        assert mm.mamba_device_status() == 0, (dim, n, l, mm.mamba_debug_build())
        for k, v in g1.items():
            assert v is None or torch.equal(g2[k], v), k
        w = oracle.scan_inputs_f64(inp)
        ref = oracle.scan_bwd(w["u"], w["delta"], w["A"], w["B"], w["C"], synth.widen(dyh, dtype),
                              dt_bias=w["dt_bias"], D_skip=w["D_skip"], z=w["z"], h0=h0,
                              dfinal=dfin)
        for gk, rk in (("du", "du"), ("dB", "dB"), ("dC", "dC"), ("dA", "dA"),
                       ("d_initial_state", "dh0")):
            got, want = to_f64(g1[gk]), ref[rk]
            if dtype == synth.F32:
                scale = max(1.0, float(np.sqrt(np.mean(want * want))))
                assert np.max(np.abs(got - want)) <= 1e-4 * scale, gk
            else:
                assert_close(got, want, dtype, gk, bf16_output=gk == "du")
    # the self-test: a check one past the end is reported, with its line
    mm.mamba_selftest_bounds()
    assert mm.mamba_device_status() == BOUNDS
    is_debug, line = mm.mamba_debug_build()
    assert is_debug and line > 0
    assert mm.mamba_device_status() == 0   # the word was cleared
    print("debug build ok")


if __name__ == "__main__":
    main()
