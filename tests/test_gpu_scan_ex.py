"""GPU parity of the extended entry points (mamba_scan_fwd_ex,
mamba_state_update_ex) against the fp64 oracle, through the C ABI.

Covers the zero-order-hold input term (with A entries equal to 0 taking the
Euler limit), a caller-supplied initial state, per-entry lengths of a padded
batch (0, full and ragged, crossing time-chunk boundaries), a long sequence
handed over in pieces (each from the previous piece's final state), a
prefill followed by generation steps, and the no-allocation flag, on the
whole-sequence, chunked and side-stream tail plans.
"""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import TOL_F32_ABS, assert_close, f32_dev, to_dev, to_f64, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_tuning():
    import selective_state_space_135_b300 as mm
    mm.mamba_scan_set_tuning(0, 0, 0)
    yield
    mm.mamba_scan_set_tuning(0, 0, 0)


def _problem(dtype, batch, dim, n, l, seed, zero_a_cols=()):
    shp = synth.ScanShape("ex", batch, dim, n, l, dtype=dtype, seed=seed)
    inp = synth.scan_inputs(shp)
    for col in zero_a_cols:
        if col < n:
            inp["A"][:, col] = 0.0
    return shp, inp


def _h0(shp, seed, scale=0.5):
    g = np.random.default_rng(seed)
    return (scale * g.standard_normal((shp.batch, shp.dim, shp.dstate))).astype(np.float32)


def _lens(batch, l, seed):
    g = np.random.default_rng(seed)
    lens = g.integers(0, l + 1, batch).astype(np.int32)
    lens[0] = l                                  # one full entry
    if batch > 1:
        lens[1] = 0                              # one empty entry
    return lens


def gpu_ex(inp, zoh=False, h0=None, lens=None, no_alloc=False, softplus=True, sl=None):
    """mamba_scan_fwd_ex on the inputs (time slice `sl` of them, if given)."""
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    dt = inp["dtype"]
    cut = (lambda a: a) if sl is None else (lambda a: np.ascontiguousarray(a[..., sl]))
    u, delta, z, B, C = (to_dev(cut(inp[k]), dt) for k in ("u", "delta", "z", "B", "C"))
    A = f32_dev(inp["A"])
    bt, d, _ = u.shape
    fin = torch.full((bt, d, A.shape[1]), float("nan"), dtype=torch.float32, device="cuda")
    h0t = None if h0 is None else (h0 if hasattr(h0, "is_cuda") else f32_dev(h0))
    lt = None if lens is None else torch.from_numpy(np.asarray(lens, np.int32)).cuda()
    y = mm.mamba_scan_fwd_ex(u, delta, f32_dev(inp["dt_bias"]), A, B, C, f32_dev(inp["D_skip"]),
                             z, softplus=softplus, zoh=zoh, initial_state=h0t, seqlens=lt,
                             final_state=fin, no_alloc=no_alloc)
    torch.cuda.synchronize()
    return y, fin


def oracle_ex(inp, zoh=False, h0=None, lens=None, softplus=True, sl=None):
    """Expected y and final state: per entry b, the oracle over its first
    lens[b] steps from h0[b]; y past lens[b] is 0."""
    w = oracle.scan_inputs_f64(inp)
    if sl is not None:
        for k in ("u", "delta", "z", "B", "C"):
            w[k] = np.ascontiguousarray(w[k][..., sl])
    bt, d, l = w["u"].shape
    n = w["A"].shape[1]
    h0d = None if h0 is None else np.asarray(h0, np.float64)
    if lens is None:
        y, hT, _ = oracle.scan(w["u"], w["delta"], w["A"], w["B"], w["C"], dt_bias=w["dt_bias"],
                               D_skip=w["D_skip"], z=w["z"], softplus=softplus, h0=h0d, zoh=zoh)
        return y, hT
    y = np.zeros((bt, d, l))
    hT = np.empty((bt, d, n))
    for b in range(bt):
        m = int(min(max(lens[b], 0), l))
        hb = None if h0d is None else h0d[b:b + 1]
        if m == 0:
            hT[b] = 0.0 if hb is None else hb[0]
            continue
        part = {k: np.ascontiguousarray(w[k][b:b + 1, :, :m]) for k in ("u", "delta", "z", "B", "C")}
        yb, hb_end, _ = oracle.scan(part["u"], part["delta"], w["A"], part["B"], part["C"],
                                    dt_bias=w["dt_bias"], D_skip=w["D_skip"], z=part["z"],
                                    softplus=softplus, h0=hb, zoh=zoh)
        y[b, :, :m] = yb[0]
        hT[b] = hb_end[0]
    return y, hT


SHAPES = [
    # dtype, batch, dim, N, L: whole units, ragged tails, dstate 4/8/16 (both splits)
    (synth.F32, 2, 33, 4, 70),
    (synth.F32, 1, 100, 16, 257),
    (synth.BF16, 2, 129, 8, 64),
    (synth.BF16, 3, 100, 16, 300),
    (synth.BF16, 2, 70, 16, 1024),
]


# --------------------------------------------------------------------------
# zero-order hold

@pytest.mark.parametrize("dtype,batch,dim,n,l", SHAPES)
def test_zoh_matches_oracle(dtype, batch, dim, n, l):
    shp, inp = _problem(dtype, batch, dim, n, l, seed=300 + l, zero_a_cols=(3,))
    y, fin = gpu_ex(inp, zoh=True)
    yr, hr = oracle_ex(inp, zoh=True)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("tail,chunks", [(0, 3), (0, 7), (2, 0), (3, 0)])
def test_zoh_chunked(dtype, tail, chunks):
    import selective_state_space_135_b300 as mm
    shp, inp = _problem(dtype, 2, 150, 16, 1000 if dtype == synth.F32 else 1024, seed=31)
    mm.mamba_scan_set_tuning(tail, 0, chunks)
    y, fin = gpu_ex(inp, zoh=True)
    yr, hr = oracle_ex(inp, zoh=True)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")


def test_theorem1_exact_under_zoh_fp32():
    # N = 1, A = -1, B = C = 1, no skip, no gate: the ZOH scan of the raw input
    # is the gated RNN h = (1 - g) h + g x with g = sigmoid(delta + dt_bias)
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    g = np.random.default_rng(1013)
    rows, l = 16, 64
    s_pre = (0.5 * g.standard_normal((1, rows, l))).astype(np.float32)
    bias = g.uniform(-4, 1, rows).astype(np.float32)
    x = g.standard_normal((1, rows, l)).astype(np.float32)
    ones = np.ones((1, 1, l), np.float32)
    y = mm.mamba_scan_fwd_ex(f32_dev(x), f32_dev(s_pre), f32_dev(bias),
                             f32_dev(-np.ones((rows, 1))), f32_dev(ones), f32_dev(ones), None,
                             None, softplus=True, zoh=True)
    torch.cuda.synchronize()
    gate = 1.0 / (1.0 + np.exp(-(s_pre.astype(np.float64) + bias[None, :, None])))
    h = np.zeros(rows)
    ref = np.empty((rows, l))
    for t in range(l):
        h = (1 - gate[0, :, t]) * h + gate[0, :, t] * x[0, :, t]
        ref[:, t] = h
    assert np.max(np.abs(to_f64(y)[0] - ref)) <= TOL_F32_ABS


# --------------------------------------------------------------------------
# initial state and per-entry lengths

@pytest.mark.parametrize("dtype,batch,dim,n,l", SHAPES)
@pytest.mark.parametrize("zoh", [False, True])
def test_initial_state(dtype, batch, dim, n, l, zoh):
    shp, inp = _problem(dtype, batch, dim, n, l, seed=400 + l)
    h0 = _h0(shp, 401)
    y, fin = gpu_ex(inp, zoh=zoh, h0=h0)
    yr, hr = oracle_ex(inp, zoh=zoh, h0=h0)
    assert_close(to_f64(y), yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")


@pytest.mark.parametrize("dtype,batch,dim,n,l", SHAPES)
@pytest.mark.parametrize("with_h0", [False, True])
def test_seqlens(dtype, batch, dim, n, l, with_h0):
    shp, inp = _problem(dtype, max(batch, 3), dim, n, l, seed=500 + l)
    lens = _lens(shp.batch, l, 501 + l)
    h0 = _h0(shp, 502) if with_h0 else None
    y, fin = gpu_ex(inp, h0=h0, lens=lens)
    yr, hr = oracle_ex(inp, h0=h0, lens=lens)
    yg = to_f64(y)
    for b in range(shp.batch):
        assert np.all(yg[b, :, lens[b]:] == 0.0), f"y past the length of entry {b}"
    assert_close(yg, yr, dtype)
    assert_close(to_f64(fin), hr, dtype, "final_state")


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("tail,chunks", [(0, 3), (0, 9), (2, 0), (3, 0)])
def test_initial_state_and_seqlens_chunked(dtype, tail, chunks):
    # lengths that end inside, at and before chunk boundaries, with a start state
    import selective_state_space_135_b300 as mm
    l = 1000 if dtype == synth.F32 else 1024
    shp, inp = _problem(dtype, 4, 150, 16, l, seed=33)
    lens = np.array([l, 0, 337, l // 3], np.int32)
    h0 = _h0(shp, 34)
    mm.mamba_scan_set_tuning(tail, 0, chunks)
    for zoh in (False, True):
        y, fin = gpu_ex(inp, zoh=zoh, h0=h0, lens=lens)
        yr, hr = oracle_ex(inp, zoh=zoh, h0=h0, lens=lens)
        assert_close(to_f64(y), yr, dtype)
        assert_close(to_f64(fin), hr, dtype, "final_state")


def test_lengths_are_clamped():
    shp, inp = _problem(synth.BF16, 3, 64, 16, 128, seed=35)
    lens = np.array([-5, 1000, 64], np.int32)
    y, fin = gpu_ex(inp, lens=lens)
    yr, hr = oracle_ex(inp, lens=np.clip(lens, 0, 128))
    assert_close(to_f64(y), yr, synth.BF16)
    assert_close(to_f64(fin), hr, synth.BF16, "final_state")


def test_zero_length_copies_initial_state():
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    u = torch.empty((2, 8, 0), dtype=torch.bfloat16, device="cuda")
    Bm = torch.empty((2, 4, 0), dtype=torch.bfloat16, device="cuda")
    A = -torch.ones((8, 4), device="cuda")
    h0 = torch.randn((2, 8, 4), device="cuda")
    fin = torch.full((2, 8, 4), 7.0, device="cuda")
    mm.mamba_scan_fwd_ex(u, u.clone(), None, A, Bm, Bm.clone(), None, None, initial_state=h0,
                         final_state=fin)
    torch.cuda.synchronize()
    assert bool((fin == h0).all())


# --------------------------------------------------------------------------
# chunked prefill and the hand-over to generation

@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("zoh", [False, True])
def test_prefill_in_pieces(dtype, zoh):
    # one 2048-step sequence handed over as pieces of 1000, 24 and 1024 steps,
    # each from the previous piece's final state
    shp, inp = _problem(dtype, 2, 200, 16, 2048, seed=36)
    yr, hr = oracle_ex(inp, zoh=zoh)
    pieces = [(0, 1000), (1000, 1024), (1024, 2048)]
    h = None
    ys = []
    for a, b in pieces:
        y, fin = gpu_ex(inp, zoh=zoh, h0=h, sl=slice(a, b))
        ys.append(to_f64(y))
        h = fin.clone()
    assert_close(np.concatenate(ys, axis=2), yr, dtype)
    assert_close(to_f64(h), hr, dtype, "final_state")


@pytest.mark.parametrize("zoh", [False, True])
def test_prefill_then_decode(zoh):
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    dtype, l0, steps = synth.BF16, 512, 24
    shp, inp = _problem(dtype, 3, 96, 16, l0 + steps, seed=37)
    yr, hr = oracle_ex(inp, zoh=zoh)
    y0, state = gpu_ex(inp, zoh=zoh, sl=slice(0, l0))
    assert_close(to_f64(y0), yr[..., :l0], dtype)
    A, dtb, dsk = f32_dev(inp["A"]), f32_dev(inp["dt_bias"]), f32_dev(inp["D_skip"])
    outs = []
    for t in range(l0, l0 + steps):
        x, dl, z, B, C = (to_dev(np.ascontiguousarray(inp[k][..., t]), dtype)
                          for k in ("u", "delta", "z", "B", "C"))
        outs.append(to_f64(mm.mamba_state_update_ex(state, x, dl, dtb, A, B, C, dsk, z,
                                                    softplus=True, zoh=zoh)))
    torch.cuda.synchronize()
    assert_close(np.stack(outs, axis=2), yr[..., l0:], dtype, "decode y")
    assert_close(to_f64(state), hr, dtype, "decode state")


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("softplus,zoh", [(False, False), (False, True), (True, True)])
def test_state_update_ex_matches_oracle(dtype, softplus, zoh):
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    g = np.random.default_rng(38)
    for batch, dim, n in ((4, 96, 16), (3, 50, 5)):
        h0 = (0.3 * g.standard_normal((batch, dim, n))).astype(np.float32)
        x = synth.store(g.standard_normal((batch, dim)).astype(np.float32), dtype)
        raw = g.standard_normal((batch, dim)).astype(np.float32)
        dl = synth.store(np.abs(raw) * 0.2 + 0.01 if not softplus else raw, dtype)
        z = synth.store(g.standard_normal((batch, dim)).astype(np.float32), dtype)
        B = synth.store(g.standard_normal((batch, n)).astype(np.float32), dtype)
        C = synth.store(g.standard_normal((batch, n)).astype(np.float32), dtype)
        A = -np.tile(np.arange(1, n + 1, dtype=np.float32), (dim, 1))
        A[:, 2] = 0.0
        dtb = (g.uniform(-4, -2, dim) if softplus else np.zeros(dim)).astype(np.float32)
        dsk = g.standard_normal(dim).astype(np.float32)
        state = f32_dev(h0)
        y = mm.mamba_state_update_ex(state, to_dev(x, dtype), to_dev(dl, dtype), f32_dev(dtb),
                                     f32_dev(A), to_dev(B, dtype), to_dev(C, dtype),
                                     f32_dev(dsk), to_dev(z, dtype), softplus=softplus, zoh=zoh)
        torch.cuda.synchronize()
        href = h0.astype(np.float64)
        yref = oracle.state_update(href, synth.widen(x, dtype), synth.widen(dl, dtype), A,
                                   synth.widen(B, dtype), synth.widen(C, dtype), dt_bias=dtb,
                                   D_skip=dsk, z=synth.widen(z, dtype), softplus=softplus, zoh=zoh)
        assert_close(to_f64(y), yref, dtype, "decode y")
        assert_close(to_f64(state), href, dtype, "decode state")


# --------------------------------------------------------------------------
# the no-allocation flag

def test_noalloc_flag_matches_oracle():
    shp, inp = _problem(synth.BF16, 2, 300, 16, 1024, seed=39)
    h0 = _h0(shp, 40)
    lens = np.array([1024, 777], np.int32)
    y, fin = gpu_ex(inp, zoh=True, h0=h0, lens=lens, no_alloc=True)
    yr, hr = oracle_ex(inp, zoh=True, h0=h0, lens=lens)
    assert_close(to_f64(y), yr, synth.BF16)
    assert_close(to_f64(fin), hr, synth.BF16, "final_state")


def test_euler_ex_equals_plain_entry_point():
    # flags = SOFTPLUS with no state and no lengths is mamba_scan_fwd, bit for bit
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    shp, inp = _problem(synth.BF16, 2, 150, 16, 512, seed=41)
    y1, f1 = gpu_ex(inp)
    dt = inp["dtype"]
    u, delta, z, B, C = (to_dev(inp[k], dt) for k in ("u", "delta", "z", "B", "C"))
    f2 = torch.empty_like(f1)
    y2 = mm.mamba_scan_fwd(u, delta, f32_dev(inp["dt_bias"]), f32_dev(inp["A"]), B, C,
                           f32_dev(inp["D_skip"]), z, True, final_state=f2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(f1, f2)


def test_extended_modes_on_a_full_wave_with_a_side_stream_tail():
    # 3 x 3200 channels are 300 tiles of 32: whole-sequence tiles on the
    # caller's stream and the 4 leftover tiles cut into time chunks on the
    # library's side stream (tail mode 3), with an initial state, per-entry
    # lengths and both discretisations
    import selective_state_space_135_b300 as mm
    shp, inp = _problem(synth.BF16, 3, 3200, 16, 1024, seed=43)
    h0 = _h0(shp, 44)
    lens = np.array([1024, 517, 800], np.int32)
    mm.mamba_scan_set_tuning(3, 0, 0)
    for zoh in (False, True):
        y, fin = gpu_ex(inp, zoh=zoh, h0=h0, lens=lens)
        yr, hr = oracle_ex(inp, zoh=zoh, h0=h0, lens=lens)
        assert_close(to_f64(y), yr, synth.BF16)
        assert_close(to_f64(fin), hr, synth.BF16, "final_state")
    assert mm.mamba_device_status() == 0
