"""GPU parity of mamba_scan_fwd against the fp64 oracle, through the C ABI.

Element-by-element on the same seeded inputs: every workload at its full size
(sampled rows where the oracle would take minutes), odd shapes with ragged
tails, every nullable argument, the chunked (summary + carry) path, both
tail scheduling modes, and guard bands around the outputs.
"""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import (TOL_F32_ABS, assert_close, f32_dev, scan_on_gpu, to_dev, to_f64,
                            torch_mod)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_tuning():
    import selective_state_space_135_b300 as mm
    mm.mamba_scan_set_tuning(0, 0, 0)
    yield
    mm.mamba_scan_set_tuning(0, 0, 0)


def oracle_full(inp, z_none=False, dskip_none=False, bias_none=False):
    w = oracle.scan_inputs_f64(inp)
    y, hT, _ = oracle.scan(w["u"], w["delta"], w["A"], w["B"], w["C"],
                           dt_bias=None if bias_none else w["dt_bias"],
                           D_skip=None if dskip_none else w["D_skip"],
                           z=None if z_none else w["z"], softplus=inp["softplus"])
    return y, hT


# --------------------------------------------------------------------------
# the five workloads

def test_tiny_fp32_full():
    inp = synth.scan_inputs(synth.TINY)
    y, fin = scan_on_gpu(inp)
    yr, hr = oracle_full(inp)
    assert_close(to_f64(y), yr, synth.F32)
    assert_close(to_f64(fin), hr, synth.F32, "final_state")
    # the workload's own bound, plain: max-abs 1e-5
    assert np.max(np.abs(to_f64(y) - yr)) <= TOL_F32_ABS
    assert np.max(np.abs(to_f64(fin) - hr)) <= TOL_F32_ABS


def test_theorem1_case_fp32():
    # N = 1, A = -1, B = C = 1, D_skip = 0, no gate: with the input rescaled by
    # g/Delta the scan must reproduce the gated RNN h = (1-g) h + g x.
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    g = np.random.default_rng(1000)
    rows, l = 16, 64
    s_pre = (0.5 * g.standard_normal((1, rows, l))).astype(np.float32)
    bias = g.uniform(-4, -2, rows).astype(np.float32)
    x = g.standard_normal((1, rows, l))
    s = s_pre.astype(np.float64) + bias[None, :, None]
    gate = 1.0 / (1.0 + np.exp(-s))
    dt = np.logaddexp(0.0, s)
    u = (x * gate / dt).astype(np.float32)
    ones = np.ones((1, 1, l), np.float32)
    y = torch.empty((1, rows, l), dtype=torch.float32, device="cuda")
    mm.mamba_scan_fwd(f32_dev(u), f32_dev(s_pre), f32_dev(bias), f32_dev(-np.ones((rows, 1))),
                      f32_dev(ones), f32_dev(ones), None, None, True, y=y)
    torch.cuda.synchronize()
    # gated RNN h = (1-g) h + g x' on the fp32-rounded input x' = u * Delta / g
    xr = u.astype(np.float64) * dt / gate
    h = np.zeros(rows)
    ref = np.empty((rows, l))
    for t in range(l):
        h = (1 - gate[0, :, t]) * h + gate[0, :, t] * xr[0, :, t]
        ref[:, t] = h
    assert np.max(np.abs(to_f64(y)[0] - ref)) <= TOL_F32_ABS


def test_m130_bf16_full():
    inp = synth.scan_inputs(synth.M130)
    y, fin = scan_on_gpu(inp)
    yr, hr = oracle_full(inp)
    st = assert_close(to_f64(y), yr, synth.BF16)
    assert_close(to_f64(fin), hr, synth.BF16, "final_state")
    print("m130", st)


def _sampled(shape, nrows, seed):
    inp = synth.scan_inputs(shape)
    y, fin = scan_on_gpu(inp)
    rows = synth.sample_rows(seed, shape.batch, shape.dim, nrows)
    ys, hs = oracle.scan_rows(inp, rows)
    yg = to_f64(y.reshape(-1, shape.seqlen)[rows])
    hg = to_f64(fin.reshape(-1, shape.dstate)[rows])
    st = assert_close(yg, ys, synth.BF16)
    assert_close(hg, hs, synth.BF16, "final_state")
    assert bool(torch_mod().isfinite(y.float()).all())
    return st


def test_m2p8_bf16_sampled_rows():
    st = _sampled(synth.M2P8, 384, 7)
    print("m2p8", st)


@pytest.mark.slow
def test_long_bf16_sampled_rows():
    st = _sampled(synth.LONG, 48, 8)
    print("long", st)


@pytest.mark.slow
def test_long1m_bf16_sampled_rows():
    """The million-step scan (the length the induction-head result on the
    pages extrapolates to): 1 x 1536 channels x 1,048,576 steps, time-chunked
    with a carry pass; 48 sampled rows against the oracle in full length,
    plus every channel of the first and the last channel tile."""
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    shp = synth.LONG1M
    small = synth.rowwise_small_inputs(shp)
    u, delta, z = (synth.rowwise_to_device(shp, k) for k in ("u", "delta", "z"))
    y = torch.empty_like(u)
    fin = torch.empty((shp.batch, shp.dim, shp.dstate), device="cuda")
    mm.mamba_scan_fwd(u, delta, f32_dev(small["dt_bias"]), f32_dev(small["A"]),
                      to_dev(small["B"], shp.dtype), to_dev(small["C"], shp.dtype),
                      f32_dev(small["D_skip"]), z, True, y=y, final_state=fin)
    torch.cuda.synchronize()
    assert mm.mamba_device_status() == 0
    rows = np.unique(np.concatenate([synth.sample_rows(9, shp.batch, shp.dim, 40),
                                     [0, 1, 31, 32, shp.dim - 33, shp.dim - 1]]))
    sub = synth.rowwise_sample(shp, rows)
    w = oracle.scan_inputs_f64(sub)
    yr, hr, _ = oracle.scan(w["u"], w["delta"], w["A"], w["B"], w["C"], dt_bias=w["dt_bias"],
                            D_skip=w["D_skip"], z=w["z"])
    assert_close(to_f64(y.reshape(-1, shp.seqlen)[rows]), yr[0], shp.dtype)
    assert_close(to_f64(fin.reshape(-1, shp.dstate)[rows]), hr[0], shp.dtype, "final_state")
    assert bool(torch.isfinite(y.float()).all())


# --------------------------------------------------------------------------
# odd shapes, ragged tails, nullable arguments

ODD = [
    # dtype, batch, dim, N, L
    (synth.F32, 1, 1, 1, 1),
    (synth.F32, 2, 33, 4, 7),
    (synth.F32, 1, 100, 16, 63),
    (synth.F32, 3, 129, 13, 65),
    (synth.F32, 1, 17, 5, 257),
    (synth.F32, 1, 40, 16, 4097),
    (synth.BF16, 1, 1, 1, 1),
    (synth.BF16, 2, 33, 3, 7),
    (synth.BF16, 1, 100, 16, 63),
    (synth.BF16, 2, 129, 8, 64),
    (synth.BF16, 3, 300, 16, 65),
    (synth.BF16, 1, 64, 2, 257),
    (synth.BF16, 2, 200, 16, 4097),
    (synth.BF16, 1, 130, 16, 4096),
]


@pytest.mark.parametrize("dtype,batch,dim,n,l", ODD)
def test_odd_shapes(dtype, batch, dim, n, l):
    shp = synth.ScanShape("odd", batch, dim, n, l, dtype=dtype, seed=77 + l + dim)
    inp = synth.scan_inputs(shp)
    y, fin = scan_on_gpu(inp)
    yr, hr = oracle_full(inp)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("z_none,dskip_none,bias_none,softplus",
                         [(True, False, False, True), (False, True, False, True),
                          (False, False, True, True), (True, True, True, True),
                          (False, False, False, False)])
def test_nullable_and_flags(dtype, z_none, dskip_none, bias_none, softplus):
    shp = synth.ScanShape("flags", 2, 70, 16, 200, dtype=dtype, softplus=softplus, seed=5)
    inp = synth.scan_inputs(shp)
    if not softplus:
        # Delta = delta + dt_bias is used as given: keep it positive and Mamba-sized
        mag = np.abs(synth.widen(inp["delta"], dtype)).astype(np.float32) * 0.2 + 0.01
        inp["delta"] = synth.store(mag, dtype)
        inp["dt_bias"] = np.linspace(0.0, 0.05, shp.dim, dtype=np.float32)
    y, fin = scan_on_gpu(inp, z_none=z_none, dskip_none=dskip_none, bias_none=bias_none)
    yr, hr = oracle_full(inp, z_none=z_none, dskip_none=dskip_none, bias_none=bias_none)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")


def test_zero_length_writes_zero_state():
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    u = torch.empty((2, 8, 0), dtype=torch.bfloat16, device="cuda")
    Bm = torch.empty((2, 4, 0), dtype=torch.bfloat16, device="cuda")
    A = -torch.ones((8, 4), device="cuda")
    fin = torch.full((2, 8, 4), 7.0, device="cuda")
    mm.mamba_scan_fwd(u, u.clone(), None, A, Bm, Bm.clone(), None, None, True, final_state=fin)
    torch.cuda.synchronize()
    assert bool((fin == 0).all())


# --------------------------------------------------------------------------
# chunked path and tail modes (same results up to fp32 rounding order)

@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("tail,chunks,stages", [(0, 3, 0), (0, 7, 3), (2, 0, 0), (1, 0, 4),
                                                (2, 5, 2), (1, 9, 1), (1, 2, 0), (2, 1, 3),
                                                (0, 1, 2)])
def test_chunks_and_tails(dtype, tail, chunks, stages):
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("chunks", 2, 150, 16, 1000 if dtype == synth.F32 else 1024,
                          dtype=dtype, seed=11)
    inp = synth.scan_inputs(shp)
    mm.mamba_scan_set_tuning(tail, stages, chunks)
    y, fin = scan_on_gpu(inp)
    yr, hr = oracle_full(inp)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")


@pytest.mark.parametrize("tail", [1, 2, 3])
def test_tail_modes_on_a_full_wave(tail):
    # 3 x 50 channel tiles of 64 fill one wave of 148 SMs with 2 tiles left
    # over: tail 2 and 3 cut those two into time chunks (3: on the side stream)
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("tail", 3, 3200, 16, 1024, seed=15)
    inp = synth.scan_inputs(shp)
    mm.mamba_scan_set_tuning(tail, 0, 0)
    y, fin = scan_on_gpu(inp)
    rows = synth.sample_rows(16, shp.batch, shp.dim, 512)
    # include every channel of the last tile (the one that is chunked)
    rows = np.unique(np.concatenate([rows, np.arange(shp.batch * shp.dim - 128, shp.batch * shp.dim)]))
    ys, hs = oracle.scan_rows(inp, rows)
    assert_close(to_f64(y.reshape(-1, shp.seqlen)[rows]), ys, shp.dtype)
    assert_close(to_f64(fin.reshape(-1, shp.dstate)[rows]), hs, shp.dtype, "final_state")
    assert mm.mamba_device_status() == 0


def test_chunk_boundary_reset():
    # A huge Delta at the first step of a chunk resets the state there; the
    # outputs after it must not depend on anything earlier, across the carry.
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("reset", 1, 64, 16, 2048, dtype=synth.F32, seed=12)
    inp = synth.scan_inputs(shp)
    mm.mamba_scan_set_tuning(0, 0, 4)          # chunks of 512 steps
    d = inp["delta"].copy()
    d[:, :, 512] = 40.0
    inp["delta"] = d
    y1, _ = scan_on_gpu(inp)
    u2 = inp["u"].copy()
    u2[:, :, :512] += 3.0
    y2, _ = scan_on_gpu(dict(inp, u=u2))
    a, b = to_f64(y1), to_f64(y2)
    assert np.max(np.abs(a[:, :, :512] - b[:, :, :512])) > 1e-2
    assert np.max(np.abs(a[:, :, 512:] - b[:, :, 512:])) <= 1e-6


# --------------------------------------------------------------------------
# guard bands: nothing outside y / final_state is written

@pytest.mark.parametrize("dtype,offset", [(synth.BF16, 8), (synth.BF16, 1), (synth.F32, 4),
                                          (synth.F32, 1)])
def test_guard_bands(dtype, offset):
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("guard", 2, 96, 16, 256 if offset % 4 == 0 else 250, dtype=dtype,
                          seed=13)
    inp = synth.scan_inputs(shp)
    tdt = torch.bfloat16 if dtype == synth.BF16 else torch.float32
    u = to_dev(inp["u"], dtype)
    n_y = u.numel()
    pad = 4096
    ybuf = torch.full((n_y + 2 * pad + offset,), -777.0, dtype=tdt, device="cuda")
    y = ybuf[pad + offset: pad + offset + n_y].view(u.shape)
    n_f = 2 * 96 * 16
    fbuf = torch.full((n_f + 2 * pad,), -555.0, device="cuda")
    fin = fbuf[pad: pad + n_f].view(2, 96, 16)
    mm.mamba_scan_fwd(u, to_dev(inp["delta"], dtype), f32_dev(inp["dt_bias"]), f32_dev(inp["A"]),
                      to_dev(inp["B"], dtype), to_dev(inp["C"], dtype), f32_dev(inp["D_skip"]),
                      to_dev(inp["z"], dtype), True, y=y, final_state=fin)
    torch.cuda.synchronize()
    assert bool((ybuf[: pad + offset] == -777.0).all())
    assert bool((ybuf[pad + offset + n_y:] == -777.0).all())
    assert bool((fbuf[:pad] == -555.0).all()) and bool((fbuf[pad + n_f:] == -555.0).all())
    yr, hr = oracle_full(inp)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")


def test_concurrent_streams_match():
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("streams", 2, 256, 16, 2048, seed=14)
    inp = synth.scan_inputs(shp)
    mm.mamba_scan_set_tuning(0, 0, 4)    # force scratch use on both streams
    args = [to_dev(inp["u"], shp.dtype), to_dev(inp["delta"], shp.dtype), f32_dev(inp["dt_bias"]),
            f32_dev(inp["A"]), to_dev(inp["B"], shp.dtype), to_dev(inp["C"], shp.dtype),
            f32_dev(inp["D_skip"]), to_dev(inp["z"], shp.dtype)]
    ref = mm.mamba_scan_fwd(*args, True)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        for s in (s1, s2):
            with torch.cuda.stream(s):
                outs.append(mm.mamba_scan_fwd(*args, True, stream=s))
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, ref)
    assert mm.mamba_device_status() == 0
