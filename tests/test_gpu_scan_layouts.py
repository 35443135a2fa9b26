"""GPU parity of both state splits of the scan kernel for dstate 9..16 against
the fp64 oracle, through the C ABI.

For dstate > 8 the library splits each channel's 16-entry state over two
warps (8 entries a lane, 64 channels per CTA) when there are enough channels,
else over four (4 a lane, 32 channels per CTA).  Each test forces one split
with the layout knob on shapes that exercise every path: dstate 9 to 16,
channel counts that leave a partial tile, sequence lengths that leave a
partial time tile, the chunked plans (summary, carry and main passes, on the
caller's stream and on the side stream), every nullable argument, the
extended modes (initial state, per-entry lengths, zero-order hold), the
no-allocation scratch, and both I/O dtypes.  Results are compared element by
element with the oracle, and the two splits with each other.
"""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, scan_on_gpu, to_f64, torch_mod
from tests.test_gpu_scan_ex import _h0, _lens, _problem, gpu_ex, oracle_ex

pytestmark = pytest.mark.gpu

SPLIT2, SPLIT4 = 1, 2


@pytest.fixture(autouse=True)
def _reset_tuning():
    import selective_state_space_135_b300 as mm
    mm.mamba_scan_set_tuning(0, 0, 0, 0)
    yield
    mm.mamba_scan_set_tuning(0, 0, 0, 0)


def _oracle(inp, z_none=False, dskip_none=False, bias_none=False):
    w = oracle.scan_inputs_f64(inp)
    y, hT, _ = oracle.scan(w["u"], w["delta"], w["A"], w["B"], w["C"],
                           dt_bias=None if bias_none else w["dt_bias"],
                           D_skip=None if dskip_none else w["D_skip"],
                           z=None if z_none else w["z"], softplus=inp["softplus"])
    return y, hT


# rows of 16 bytes (tensor-map path): bf16 seqlen % 8 == 0, fp32 seqlen % 4 == 0
SHAPES = [
    (synth.F32, 1, 100, 16, 64),
    (synth.F32, 3, 129, 13, 68),
    (synth.F32, 1, 40, 9, 1028),
    (synth.BF16, 1, 100, 16, 64),
    (synth.BF16, 3, 300, 16, 72),
    (synth.BF16, 2, 200, 12, 4096),
    (synth.BF16, 1, 130, 16, 4104),
    (synth.BF16, 2, 256, 10, 8),
]


@pytest.mark.parametrize("layout", [SPLIT2, SPLIT4])
@pytest.mark.parametrize("dtype,batch,dim,n,l", SHAPES)
def test_split_shapes(dtype, batch, dim, n, l, layout):
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("layouts", batch, dim, n, l, dtype=dtype, seed=91 + l + dim)
    inp = synth.scan_inputs(shp)
    mm.mamba_scan_set_tuning(0, 0, 0, layout)
    y, fin = scan_on_gpu(inp)
    yr, hr = _oracle(inp)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")
    assert mm.mamba_device_status() == 0


@pytest.mark.parametrize("layout", [SPLIT2, SPLIT4])
@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("tail,chunks,stages", [(0, 3, 0), (0, 7, 2), (2, 0, 0), (1, 0, 4),
                                                (2, 5, 2), (1, 2, 3), (0, 1, 0)])
def test_split_chunks_and_stages(dtype, tail, chunks, stages, layout):
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("split chunks", 2, 250, 16, 1000 if dtype == synth.F32 else 1024,
                          dtype=dtype, seed=21)
    inp = synth.scan_inputs(shp)
    mm.mamba_scan_set_tuning(tail, stages, chunks, layout)
    y, fin = scan_on_gpu(inp)
    yr, hr = _oracle(inp)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")
    assert mm.mamba_device_status() == 0


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("z_none,dskip_none,bias_none,softplus",
                         [(True, False, False, True), (False, True, False, True),
                          (False, False, True, True), (True, True, True, True),
                          (False, False, False, False)])
@pytest.mark.parametrize("layout", [SPLIT2, SPLIT4])
def test_split_nullable_and_flags(dtype, z_none, dskip_none, bias_none, softplus, layout):
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("split flags", 2, 170, 16, 200, dtype=dtype, softplus=softplus, seed=6)
    inp = synth.scan_inputs(shp)
    if not softplus:
        mag = np.abs(synth.widen(inp["delta"], dtype)).astype(np.float32) * 0.2 + 0.01
        inp["delta"] = synth.store(mag, dtype)
        inp["dt_bias"] = np.linspace(0.0, 0.05, shp.dim, dtype=np.float32)
    mm.mamba_scan_set_tuning(0, 0, 0, layout)
    y, fin = scan_on_gpu(inp, z_none=z_none, dskip_none=dskip_none, bias_none=bias_none)
    yr, hr = _oracle(inp, z_none=z_none, dskip_none=dskip_none, bias_none=bias_none)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("zoh,with_h0,with_lens,chunks", [
    (True, False, False, 0), (False, True, False, 0), (False, False, True, 0),
    (True, True, True, 0), (False, True, True, 5), (True, True, False, 3)])
@pytest.mark.parametrize("layout", [SPLIT2, SPLIT4])
def test_split_extended_modes(dtype, zoh, with_h0, with_lens, chunks, layout):
    import selective_state_space_135_b300 as mm
    l = 1000 if dtype == synth.F32 else 1024
    shp, inp = _problem(dtype, 3, 200, 16, l, seed=400 + chunks, zero_a_cols=(5,))
    h0 = _h0(shp, 41) if with_h0 else None
    lens = _lens(shp.batch, l, 42) if with_lens else None
    mm.mamba_scan_set_tuning(0, 0, chunks, layout)
    y, fin = gpu_ex(inp, zoh=zoh, h0=h0, lens=lens)
    yr, hr = oracle_ex(inp, zoh=zoh, h0=h0, lens=lens)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")
    assert mm.mamba_device_status() == 0


@pytest.mark.parametrize("layout", [SPLIT2, SPLIT4])
@pytest.mark.parametrize("chunks", [0, 4])
def test_split_no_alloc(chunks, layout):
    import selective_state_space_135_b300 as mm
    shp, inp = _problem(synth.BF16, 2, 300, 16, 2048, seed=55)
    mm.mamba_scan_set_tuning(0, 0, chunks, layout)
    y, fin = gpu_ex(inp, no_alloc=True)
    yr, hr = oracle_ex(inp)
    assert_close(to_f64(y), yr, synth.BF16)
    assert_close(to_f64(fin), hr, synth.BF16, "final_state")


@pytest.mark.parametrize("tail", [1, 2, 3])
def test_split_tail_modes_on_a_full_wave(tail):
    # 3 x 100 tiles of 64 channels: two per SM of a 148-SM GPU plus 4 left
    # over, which tail 2 and 3 cut into time chunks (3: on the side stream)
    import selective_state_space_135_b300 as mm
    shp = synth.ScanShape("split tail", 3, 6400, 16, 1024, seed=16)
    inp = synth.scan_inputs(shp)
    mm.mamba_scan_set_tuning(tail, 0, 0, SPLIT2)
    y, fin = scan_on_gpu(inp)
    rows = synth.sample_rows(17, shp.batch, shp.dim, 512)
    rows = np.unique(np.concatenate(
        [rows, np.arange(shp.batch * shp.dim - 256, shp.batch * shp.dim)]))
    ys, hs = oracle.scan_rows(inp, rows)
    assert_close(to_f64(y.reshape(-1, shp.seqlen)[rows]), ys, shp.dtype)
    assert_close(to_f64(fin.reshape(-1, shp.dstate)[rows]), hs, shp.dtype, "final_state")
    assert mm.mamba_device_status() == 0


def test_two_and_four_way_splits_agree():
    # The two splits differ only in fp32 summation order: their outputs
    # agree to far inside the parity tolerance on the Mamba-130M layer shape.
    import selective_state_space_135_b300 as mm
    shp = synth.M130
    inp = synth.scan_inputs(shp)
    out = {}
    for layout in (SPLIT2, SPLIT4):
        mm.mamba_scan_set_tuning(0, 0, 0, layout)
        out[layout] = scan_on_gpu(inp)
    ya, yb = to_f64(out[SPLIT2][0]), to_f64(out[SPLIT4][0])
    rms = float(np.sqrt(np.mean(yb * yb)))
    assert float(np.sqrt(np.mean((ya - yb) ** 2))) / rms <= 2e-3
    fa, fb = to_f64(out[SPLIT2][1]), to_f64(out[SPLIT4][1])
    assert float(np.max(np.abs(fa - fb))) <= 1e-3 * float(np.sqrt(np.mean(fb * fb)))
    assert bool(torch_mod().isfinite(out[SPLIT2][0].float()).all())
