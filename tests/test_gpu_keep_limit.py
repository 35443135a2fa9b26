"""The method's keep and reset limits on the GPU (page "Mamba: linear-time
sequence modeling with selective state spaces", "Main results (verified)": a
small Delta keeps the state and ignores the input, a large Delta resets it).

Steps with delta + dt_bias far below zero give Delta = softplus(s) = e^s to
within e^2s; the bf16 path computes softplus from hardware exponentials, and
these tests hold it, element by element, to the fp64 oracle there:

  * scans with dt_bias ~ U(-20, -10), no skip term and no gate, so that y is
    C.h with h = sum of Delta*B*u and carries any relative error of Delta
    undiluted: both state splits, both dtypes, whole-sequence and chunked
    plans, and the generation step;
  * keep: from a non-zero initial state, 64 steps with s = -30 leave the
    state as it was, so y_t = C_t . h0 element by element;
  * reset: a step with a huge Delta at a chunk boundary makes every later
    output independent of every earlier input, on the bf16 path too.
"""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import BF16_UNIT_ROUNDOFF, assert_close, f32_dev, scan_on_gpu, to_dev, \
    to_f64, torch_mod
from tests.test_gpu_scan_ex import gpu_ex, oracle_ex

pytestmark = pytest.mark.gpu

SPLIT2, SPLIT4 = 1, 2


@pytest.fixture(autouse=True)
def _reset_tuning():
    import selective_state_space_135_b300 as mm
    mm.mamba_scan_set_tuning(0, 0, 0, 0)
    yield
    mm.mamba_scan_set_tuning(0, 0, 0, 0)


def _small_delta_inputs(dtype, batch, dim, n, l, seed):
    shp = synth.ScanShape("keep", batch, dim, n, l, dtype=dtype, dt_lo=-20.0, dt_hi=-10.0,
                          seed=seed)
    return shp, synth.scan_inputs(shp)


def _oracle_plain(inp):
    w = oracle.scan_inputs_f64(inp)
    y, hT, _ = oracle.scan(w["u"], w["delta"], w["A"], w["B"], w["C"], dt_bias=w["dt_bias"],
                           D_skip=None, z=None, softplus=True)
    return y, hT


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("layout,chunks", [(SPLIT2, 0), (SPLIT4, 0), (SPLIT2, 4), (SPLIT4, 4)])
def test_small_delta_scan(dtype, layout, chunks):
    import selective_state_space_135_b300 as mm
    shp, inp = _small_delta_inputs(dtype, 2, 160, 16, 1024, seed=71)
    mm.mamba_scan_set_tuning(0, 0, chunks, layout)
    y, fin = scan_on_gpu(inp, z_none=True, dskip_none=True)
    yr, hr = _oracle_plain(inp)
    # the regime really is the keep limit: Delta between about e^-25 and e^-7
    s = synth.widen(inp["delta"], dtype) + inp["dt_bias"][None, :, None]
    assert s.max() < -7.0 and s.min() > -25.0
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_small_delta_generation_steps(dtype):
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    shp, inp = _small_delta_inputs(dtype, 2, 64, 16, 48, seed=72)
    state = torch.zeros((2, 64, 16), device="cuda")
    ys = []
    for t in range(shp.seqlen):
        step = {k: np.ascontiguousarray(inp[k][..., t]) for k in ("u", "delta", "B", "C")}
        ys.append(mm.mamba_state_update(state, to_dev(step["u"], dtype),
                                        to_dev(step["delta"], dtype), f32_dev(inp["dt_bias"]),
                                        f32_dev(inp["A"]), to_dev(step["B"], dtype),
                                        to_dev(step["C"], dtype), None, None))
    torch.cuda.synchronize()
    y = torch.stack(ys, dim=-1)
    yr, hr = _oracle_plain(inp)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(state), hr, dtype, "state")


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("layout", [SPLIT2, SPLIT4])
def test_keep_from_initial_state(dtype, layout):
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("keep h0", 2, 130, 16, 64, dtype=dtype, seed=73)
    inp = synth.scan_inputs(shp)
    inp["delta"] = synth.store(np.full(inp["u"].shape, -30.0, np.float32), dtype)
    inp["dt_bias"] = np.zeros(shp.dim, np.float32)
    inp["D_skip"] = np.zeros(shp.dim, np.float32)
    inp["z"] = None
    g = np.random.default_rng(74)
    h0 = (0.5 * g.standard_normal((shp.batch, shp.dim, shp.dstate))).astype(np.float32)
    mm.mamba_scan_set_tuning(0, 0, 0, layout)
    torch = torch_mod()
    u, dl, B, C = (to_dev(inp[k], dtype) for k in ("u", "delta", "B", "C"))
    fin = torch.empty((shp.batch, shp.dim, shp.dstate), device="cuda")
    y = mm.mamba_scan_fwd_ex(u, dl, None, f32_dev(inp["A"]), B, C, None, None, softplus=True,
                             initial_state=f32_dev(h0), final_state=fin)
    torch.cuda.synchronize()
    # closed form: y[b, d, t] = sum_n C[b, n, t] h0[b, d, n]; the state stays h0
    Cw = synth.widen(inp["C"], dtype)
    ref = np.einsum("bnt,bdn->bdt", Cw, h0.astype(np.float64))
    got = to_f64(y)
    rms = float(np.sqrt(np.mean(ref * ref)))
    tol_round = BF16_UNIT_ROUNDOFF if dtype == synth.BF16 else 0.0
    assert np.max(np.abs(got - ref) - tol_round * np.abs(ref)) <= 1e-5 * rms
    assert np.max(np.abs(to_f64(fin) - h0)) <= 1e-6
    yr, hr = oracle_ex(inp, h0=h0)
    assert_close(got, yr, dtype)


@pytest.mark.parametrize("layout", [SPLIT2, SPLIT4])
def test_chunk_boundary_reset_bf16(layout):
    # A huge Delta at the first step of a chunk resets the state there; the
    # bf16 outputs after it must not depend on anything earlier, across the carry.
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("reset bf16", 1, 128, 16, 2048, seed=75)
    inp = synth.scan_inputs(shp)
    mm.mamba_scan_set_tuning(0, 0, 4, layout)   # chunks of 512 steps
    d = synth.widen(inp["delta"], synth.BF16).astype(np.float32)
    d[:, :, 512] = 40.0
    inp["delta"] = synth.store(d, synth.BF16)
    y1, _ = scan_on_gpu(inp)
    u2 = synth.widen(inp["u"], synth.BF16).astype(np.float32)
    u2[:, :, :512] += 3.0
    y2, _ = scan_on_gpu(dict(inp, u=synth.store(u2, synth.BF16)))
    a, b = to_f64(y1), to_f64(y2)
    assert np.max(np.abs(a[:, :, :512] - b[:, :, :512])) > 1e-2
    assert np.max(np.abs(a[:, :, 512:] - b[:, :, 512:])) <= 1e-6
    yr, _ = oracle_ex(inp)
    assert_close(a, yr, synth.BF16)
