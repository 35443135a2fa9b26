"""Pins for the fp64 oracle, from what the pages and the mathematics fix.

None of these re-type the oracle's loop.  Each check uses an independent
formulation or a closed form, chosen so that a plausible slip in the oracle
(a dropped term, a sign, a swapped B/C, a wrong index or layout) fails one:

* hand-worked example (tests/golden/hand_scan_n1_l3.txt);
* softplus / silu identities;
* Theorem 1 ("Mamba: linear-time sequence modeling with selective state
  spaces", "Main results": with N = 1, A = -1, B = 1 the selective SSM is the
  gated RNN h_t = (1 - g_t) h_{t-1} + g_t x_t, g_t = sigmoid(Linear(x_t))),
  in three parts: the decay equals 1 - g exactly, a rescaled input gives the
  gated RNN exactly, and the unrescaled gap shrinks like Delta^2;
* keep / reset (same page: a small Delta keeps the state, a large Delta
  resets it);
* the explicitly unrolled sum over earlier tokens (the "attention-driven"
  view on page "Mamba models"), evaluated as an O(L^2) sum in long double;
* the time-invariant special case as a causal convolution (page "Mamba:
  Linear-Time Sequence Modeling with Selective State Spaces", "Selective
  state spaces": earlier SSMs use one fixed rule; with it the model is a
  convolution), checked with numpy.convolve;
* linearity in u, causality, chunk associativity through the initial-state
  argument, decode == scan, thread-count independence;
* the zero-order-hold input term (the textbook exact discretisation of
  h' = A h + B x with x held over the step; the pages print only
  Abar = exp(Delta A)): its weight against a 50-digit evaluation, Theorem 1
  holding exactly with the unscaled input, the continuous-time steady state
  -B u / A reached exactly under constant input, the unrolled sum and the
  time-invariant convolution with the ZOH weight, and the Euler limit at
  A = 0.
"""

import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(seed, bt=2, d=3, n=4, l=40, gate=True, dskip=True, bias=True):
    g = np.random.default_rng(seed)
    return dict(
        u=g.standard_normal((bt, d, l)),
        delta=0.5 * g.standard_normal((bt, d, l)),
        z=g.standard_normal((bt, d, l)) if gate else None,
        B=g.standard_normal((bt, n, l)),
        C=g.standard_normal((bt, n, l)),
        A=-(g.uniform(0.5, 4.0, (d, n))),
        dt_bias=g.uniform(-4, -2, d) if bias else None,
        D_skip=g.standard_normal(d) if dskip else None,
    )


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            vals[k] = np.array([float(x) for x in v])
    return vals


# --------------------------------------------------------------------------

def test_hand_worked_example():
    g = _golden("hand_scan_n1_l3.txt")
    shp = lambda a: a.reshape(1, 1, -1)
    y, hT, _ = oracle.scan(shp(g["u"]), shp(g["delta"]), g["A"].reshape(1, 1),
                           shp(g["B"]), shp(g["C"]), D_skip=g["D_skip"], softplus=False)
    np.testing.assert_allclose(y.ravel(), g["y"], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(hT.ravel(), g["final"], rtol=1e-15, atol=1e-15)
    y2, hT2, _ = oracle.scan(shp(g["u"]), shp(g["delta"]), g["A"].reshape(1, 1),
                             shp(g["B"]), shp(g["C"]), D_skip=g["D_skip"],
                             z=shp(g["z_gate"]), softplus=False)
    np.testing.assert_array_equal(y2.ravel(), g["y_gated"])
    np.testing.assert_allclose(hT2.ravel(), g["final"], rtol=1e-15)


def test_softplus_silu_identities():
    for s in [-50.0, -30.0, -7.5, -1.0, -1e-3, 0.0, 1e-3, 0.7, 5.0, 30.0, 60.0]:
        sp = oracle.softplus(s)
        # softplus(s) - softplus(-s) = s ; softplus(0) = ln 2 ; e^{-softplus(s)} = sigmoid(-s)
        assert abs((sp - oracle.softplus(-s)) - s) <= 4e-16 * max(1.0, abs(s))
        assert math.isclose(math.exp(-sp), expit(-s), rel_tol=1e-14, abs_tol=1e-300)
        assert math.isclose(sp, np.logaddexp(0.0, s), rel_tol=1e-15)
        z = s / 3.0
        # silu(z) - silu(-z) = z ; silu(z) = z * sigmoid(z)
        assert math.isclose(oracle.silu(z) - oracle.silu(-z), z, rel_tol=1e-14, abs_tol=1e-15)
        assert math.isclose(oracle.silu(z), z * expit(z), rel_tol=1e-14, abs_tol=1e-300)
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-16)


# --------------------------------------------------------------------------
# Theorem 1: selection is gating

def _theorem1_inputs(seed, rows=64, l=48, bias_lo=-4.0, bias_hi=2.0):
    g = np.random.default_rng(seed)
    s_pre = g.standard_normal((rows, 1, l))
    bias = g.uniform(bias_lo, bias_hi, 1)
    x = g.standard_normal((rows, 1, l))
    return s_pre, bias, x


def test_theorem1_decay_is_one_minus_gate():
    # h0 = 1, u = 0, C = 1: y_t = prod_{s<=t} Abar_s; at t = 0 it is Abar_0 itself.
    s = np.linspace(-40.0, 40.0, 401).reshape(-1, 1, 1)
    rows = s.shape[0]
    ones = np.ones((rows, 1, 1))
    y, _, _ = oracle.scan(np.zeros((rows, 1, 1)), s, -np.ones((1, 1)), ones, ones,
                          h0=np.ones((rows, 1, 1)), softplus=True)
    gate = expit(s.ravel())
    # 1 - g loses digits to cancellation once g ~ 1, hence the absolute bound;
    # sigmoid(-s) = 1 - g exactly and carries full relative precision.
    np.testing.assert_allclose(y.ravel(), 1.0 - gate, rtol=0, atol=4e-16)
    np.testing.assert_allclose(y.ravel(), expit(-s.ravel()), rtol=2e-14, atol=1e-300)


def test_theorem1_rescaled_input_is_gated_rnn():
    s_pre, bias, x = _theorem1_inputs(7)
    rows, _, l = x.shape
    s = s_pre + bias[0]
    gate = expit(s)
    dt = -np.log1p(-gate)            # = softplus(s), written via the gate
    u_resc = x * gate / dt
    ones = np.ones((rows, 1, l))
    y, hT, _ = oracle.scan(u_resc, s_pre, -np.ones((1, 1)), ones, ones,
                           dt_bias=bias, softplus=True)
    # gated RNN, written independently
    h = np.zeros(rows)
    ref = np.empty((rows, l))
    for t in range(l):
        h = (1.0 - gate[:, 0, t]) * h + gate[:, 0, t] * x[:, 0, t]
        ref[:, t] = h
    np.testing.assert_allclose(y[:, 0, :], ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hT[:, 0, 0], ref[:, -1], rtol=1e-12, atol=1e-13)


def test_theorem1_euler_gap_is_second_order():
    # Without the rescale the input weight is Delta = -ln(1-g) = g + g^2/2 + ...
    # so over a short sequence the gap to the gated RNN is O(Delta^2).
    g = np.random.default_rng(11)
    l = 8
    s_pre = 0.3 * g.standard_normal((16, 1, l))
    x = g.standard_normal((16, 1, l))
    ones = np.ones((16, 1, l))
    errs, dts = [], []
    for bias in [-4.0, -5.0, -6.0, -7.0, -8.0]:
        y, _, _ = oracle.scan(x, s_pre, -np.ones((1, 1)), ones, ones,
                              dt_bias=np.array([bias]), softplus=True)
        gate = expit(s_pre + bias)
        h = np.zeros(16)
        ref = np.empty((16, l))
        for t in range(l):
            h = (1.0 - gate[:, 0, t]) * h + gate[:, 0, t] * x[:, 0, t]
            ref[:, t] = h
        errs.append(np.max(np.abs(y[:, 0, :] - ref)))
        dts.append(np.mean(np.logaddexp(0.0, s_pre + bias)))
    slope = np.polyfit(np.log(dts), np.log(errs), 1)[0]
    assert 1.8 < slope < 2.2, slope


# --------------------------------------------------------------------------
# keep / reset

def test_small_delta_keeps_state():
    p = _rand_problem(3, gate=False)
    bt, d, l = p["u"].shape
    n = p["A"].shape[1]
    h0 = np.random.default_rng(4).standard_normal((bt, d, n))
    # Delta = softplus(-40) ~ 4.2e-18: over L = 40 steps with |A| <= 4 the state
    # moves by at most ~L*|A|*Delta*|h| + L*Delta*|B u| ~ 1e-15
    delta = np.full_like(p["u"], -40.0)
    y, hT, _ = oracle.scan(p["u"], delta, p["A"], p["B"], p["C"], D_skip=p["D_skip"],
                           h0=h0, softplus=True)
    np.testing.assert_allclose(hT, h0, rtol=0, atol=1e-13)
    # y_t = C_t . h0 + D u_t
    expect = np.einsum("bnl,bdn->bdl", p["C"], h0) + p["D_skip"][None, :, None] * p["u"]
    np.testing.assert_allclose(y, expect, rtol=0, atol=1e-13)


def test_large_delta_resets_state():
    p = _rand_problem(5, l=48)
    n = p["A"].shape[1]
    A = -(np.arange(n, dtype=np.float64) + 1.0) * np.ones((p["A"].shape[0], 1))
    t0 = 20
    delta = p["delta"].copy()
    delta[:, :, t0] = 30.0 + 4.0                  # s = delta + bias >= 30 at t0
    y1, _, _ = oracle.scan(p["u"], delta, A, p["B"], p["C"], dt_bias=p["dt_bias"],
                           D_skip=p["D_skip"], z=p["z"])
    g = np.random.default_rng(6)
    u2 = p["u"].copy()
    u2[:, :, :t0] += 10.0 * g.standard_normal(u2[:, :, :t0].shape)
    d2 = delta.copy()
    d2[:, :, :t0] += g.standard_normal(d2[:, :, :t0].shape)
    y2, _, _ = oracle.scan(u2, d2, A, p["B"], p["C"], dt_bias=p["dt_bias"],
                           D_skip=p["D_skip"], z=p["z"])
    assert np.max(np.abs(y1[:, :, :t0] - y2[:, :, :t0])) > 1e-3   # history did matter
    np.testing.assert_allclose(y1[:, :, t0:], y2[:, :, t0:], rtol=0, atol=1e-9)


# --------------------------------------------------------------------------
# explicit unrolled sum (brute force, long double)

def _unrolled(p, softplus=True, zoh=False):
    ld = np.longdouble
    u, delta, B, C, A = (np.asarray(p[k], dtype=ld) for k in ("u", "delta", "B", "C", "A"))
    bt, d, l = u.shape
    s = delta + (np.asarray(p["dt_bias"], dtype=ld)[None, :, None] if p["dt_bias"] is not None else 0)
    if softplus:
        dt = np.log1p(np.exp(-np.abs(s))) + np.maximum(s, 0)
    else:
        dt = s
    S = np.cumsum(dt, axis=2)                     # S_T = sum_{s<=T} Delta_s
    y = np.empty((bt, d, l), dtype=ld)
    hT = np.empty((bt, d, A.shape[1]), dtype=ld)
    for T in range(l):
        # decay from step t to T: exp(A_n * sum_{s=t+1..T} Delta_s) = exp(A_n (S_T - S_t))
        gap = S[:, :, T:T + 1] - S[:, :, :T + 1]                          # (bt,d,T+1)
        w = np.exp(A[None, :, :, None] * gap[:, :, None, :])              # (bt,d,n,T+1)
        if zoh:
            # (exp(Delta A) - 1) / A per entry, written with expm1 in long double
            wt = np.expm1(A[None, :, :, None] * dt[:, :, None, :T + 1]) / A[None, :, :, None]
        else:
            wt = dt[:, :, None, :T + 1]
        drive = wt * B[:, None, :, :T + 1] * u[:, :, None, :T + 1]
        h = np.sum(w * drive, axis=3)                                     # (bt,d,n)
        y[:, :, T] = np.einsum("bdn,bn->bd", h, C[:, :, T])
        if T == l - 1:
            hT = h
    if p["D_skip"] is not None:
        y = y + np.asarray(p["D_skip"], dtype=ld)[None, :, None] * u
    if p["z"] is not None:
        z = np.asarray(p["z"], dtype=ld)
        y = y * z / (1 + np.exp(-z))
    return y.astype(np.float64), hT.astype(np.float64)


@pytest.mark.parametrize("seed,gate,dskip,bias,zoh", [
    (0, True, True, True, False), (1, False, True, True, False),
    (2, True, False, False, False), (3, False, False, True, False),
    (4, True, True, True, True), (5, False, False, True, True)])
def test_unrolled_sum_matches(seed, gate, dskip, bias, zoh):
    p = _rand_problem(seed, bt=2, d=3, n=5, l=64, gate=gate, dskip=dskip, bias=bias)
    y, hT, _ = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], dt_bias=p["dt_bias"],
                           D_skip=p["D_skip"], z=p["z"], zoh=zoh)
    yr, hr = _unrolled(p, zoh=zoh)
    scale = max(1.0, np.max(np.abs(yr)))
    np.testing.assert_allclose(y, yr, rtol=0, atol=1e-12 * scale)
    np.testing.assert_allclose(hT, hr, rtol=0, atol=1e-12 * max(1.0, np.max(np.abs(hr))))


def test_unrolled_sum_on_tiny_workload():
    inp = synth.scan_inputs(synth.TINY)
    w = oracle.scan_inputs_f64(inp)
    y, hT, _ = oracle.scan(w["u"], w["delta"], w["A"], w["B"], w["C"], dt_bias=w["dt_bias"],
                           D_skip=w["D_skip"], z=w["z"])
    yr, hr = _unrolled(w)
    np.testing.assert_allclose(y, yr, rtol=0, atol=1e-12)
    np.testing.assert_allclose(hT, hr, rtol=0, atol=1e-12)


def test_softplus_off_unrolled():
    p = _rand_problem(9, gate=True)
    p["delta"] = np.abs(p["delta"]) + 0.01        # Delta > 0 used directly
    p["dt_bias"] = None
    y, hT, _ = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], D_skip=p["D_skip"],
                           z=p["z"], softplus=False)
    yr, hr = _unrolled(p, softplus=False)
    np.testing.assert_allclose(y, yr, rtol=0, atol=1e-12 * max(1, np.abs(yr).max()))


# --------------------------------------------------------------------------
# time-invariant case == causal convolution

def test_lti_case_is_convolution():
    g = np.random.default_rng(21)
    n, l = 6, 80
    dt = 0.37
    A = -g.uniform(0.2, 3.0, (1, n))
    Bn = g.standard_normal(n)
    Cn = g.standard_normal(n)
    u = g.standard_normal((1, 1, l))
    B = np.repeat(Bn[None, :, None], l, axis=2)
    C = np.repeat(Cn[None, :, None], l, axis=2)
    delta = np.full((1, 1, l), dt)
    dsk = np.array([0.8])
    y, _, _ = oracle.scan(u, delta, A, B, C, D_skip=dsk, softplus=False)
    k = np.arange(l)
    K = np.sum(Cn[:, None] * np.exp(np.outer(A[0], k) * dt) * dt * Bn[:, None], axis=0)
    ref = np.convolve(u[0, 0], K)[:l] + dsk[0] * u[0, 0]
    np.testing.assert_allclose(y[0, 0], ref, rtol=0, atol=1e-12 * max(1, np.abs(ref).max()))


def test_lti_case_is_convolution_zoh():
    # same system, zero-order hold: K_k = sum_n C_n e^{k dt A_n} (e^{dt A_n} - 1) / A_n B_n
    g = np.random.default_rng(22)
    n, l = 5, 70
    dt = 0.29
    A = -g.uniform(0.2, 3.0, (1, n))
    Bn = g.standard_normal(n)
    Cn = g.standard_normal(n)
    u = g.standard_normal((1, 1, l))
    B = np.repeat(Bn[None, :, None], l, axis=2)
    C = np.repeat(Cn[None, :, None], l, axis=2)
    y, _, _ = oracle.scan(u, np.full((1, 1, l), dt), A, B, C, softplus=False, zoh=True)
    k = np.arange(l)
    wz = (np.exp(dt * A[0]) - 1.0) / A[0]
    K = np.sum(Cn[:, None] * np.exp(np.outer(A[0], k) * dt) * (wz * Bn)[:, None], axis=0)
    ref = np.convolve(u[0, 0], K)[:l]
    np.testing.assert_allclose(y[0, 0], ref, rtol=0, atol=1e-12 * max(1, np.abs(ref).max()))


# --------------------------------------------------------------------------
# zero-order hold

def test_zoh_weight_against_high_precision():
    import mpmath
    mpmath.mp.dps = 50
    for dt in (1e-9, 1e-4, 0.0025, 0.049, 0.7, 3.0, 40.0):
        for a in (-16.0, -1.0, -1e-3, -1e-12, 0.5, 2.0):
            exact = (mpmath.exp(mpmath.mpf(dt) * a) - 1) / a
            got = oracle.zoh_weight(dt, a)
            assert abs(got - float(exact)) <= 4e-16 * abs(float(exact)), (dt, a, got)
    # A == 0 is the limit dt; the weight never exceeds dt for A < 0
    assert oracle.zoh_weight(0.37, 0.0) == 0.37
    assert oracle.zoh_weight(0.37, -2.0) < 0.37


def test_theorem1_exact_under_zoh():
    # N = 1, A = -1, B = 1: Abar = 1 - g and the ZOH input weight is
    # (1 - e^{-Delta}) = g, so the scan is the gated RNN on the raw input.
    s_pre, bias, x = _theorem1_inputs(13)
    rows, _, l = x.shape
    gate = expit(s_pre + bias[0])
    ones = np.ones((rows, 1, l))
    y, hT, _ = oracle.scan(x, s_pre, -np.ones((1, 1)), ones, ones, dt_bias=bias,
                           softplus=True, zoh=True)
    h = np.zeros(rows)
    ref = np.empty((rows, l))
    for t in range(l):
        h = (1.0 - gate[:, 0, t]) * h + gate[:, 0, t] * x[:, 0, t]
        ref[:, t] = h
    np.testing.assert_allclose(y[:, 0, :], ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hT[:, 0, 0], ref[:, -1], rtol=1e-12, atol=1e-13)


def test_zoh_reaches_continuous_steady_state():
    # Under constant input the ZOH recurrence has the fixed point of the
    # continuous system, h = -B u / A (Euler's is Delta B u / (1 - e^{Delta A})).
    # (the residual after L steps is prod Abar = e^{-Delta |A| L} <= e^{-50} here)
    g = np.random.default_rng(17)
    n, l = 4, 2000
    A = -g.uniform(0.5, 4.0, (1, n))
    Bn = g.standard_normal(n)
    uval = 1.3
    for dt in (0.05, 0.6):
        delta = np.full((1, 1, l), dt)
        B = np.repeat(Bn[None, :, None], l, axis=2)
        C = np.zeros((1, n, l))
        _, hT, _ = oracle.scan(np.full((1, 1, l), uval), delta, A, B, C, softplus=False,
                               zoh=True)
        np.testing.assert_allclose(hT[0, 0], -Bn * uval / A[0], rtol=1e-12)
        _, hE, _ = oracle.scan(np.full((1, 1, l), uval), delta, A, B, C, softplus=False)
        assert np.max(np.abs(hE[0, 0] + Bn * uval / A[0])) > 1e-3   # Euler's differs


def test_zoh_at_zero_A_is_euler():
    p = _rand_problem(23)
    A = np.zeros_like(p["A"])
    kw = dict(dt_bias=p["dt_bias"], D_skip=p["D_skip"], z=p["z"])
    y1, h1, _ = oracle.scan(p["u"], p["delta"], A, p["B"], p["C"], zoh=True, **kw)
    y0, h0, _ = oracle.scan(p["u"], p["delta"], A, p["B"], p["C"], **kw)
    np.testing.assert_array_equal(y1, y0)
    np.testing.assert_array_equal(h1, h0)


# --------------------------------------------------------------------------
# invariants

def test_linear_in_u():
    p = _rand_problem(31)
    g = np.random.default_rng(32)
    u2 = g.standard_normal(p["u"].shape)
    a, b = 1.7, -0.6
    kw = dict(dt_bias=p["dt_bias"], D_skip=p["D_skip"], z=p["z"])
    y1, h1, _ = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], **kw)
    y2, h2, _ = oracle.scan(u2, p["delta"], p["A"], p["B"], p["C"], **kw)
    y3, h3, _ = oracle.scan(a * p["u"] + b * u2, p["delta"], p["A"], p["B"], p["C"], **kw)
    np.testing.assert_allclose(y3, a * y1 + b * y2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(h3, a * h1 + b * h2, rtol=0, atol=1e-12)


def test_causal():
    p = _rand_problem(41)
    t1 = 17
    q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
    g = np.random.default_rng(42)
    for k in ("u", "delta", "z", "B", "C"):
        q[k][..., t1 + 1:] += g.standard_normal(q[k][..., t1 + 1:].shape)
    kw = lambda r: dict(dt_bias=r["dt_bias"], D_skip=r["D_skip"], z=r["z"])
    y1, _, _ = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], **kw(p))
    y2, _, _ = oracle.scan(q["u"], q["delta"], q["A"], q["B"], q["C"], **kw(q))
    np.testing.assert_array_equal(y1[..., :t1 + 1], y2[..., :t1 + 1])
    assert np.max(np.abs(y1[..., t1 + 1:] - y2[..., t1 + 1:])) > 1e-3


def test_chunk_associativity():
    p = _rand_problem(51, l=60)
    kw = dict(dt_bias=p["dt_bias"], D_skip=p["D_skip"])
    y, hT, _ = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], z=p["z"], **kw)
    c = 23
    sl = lambda a, s: None if a is None else np.ascontiguousarray(a[..., s])
    ya, ha, _ = oracle.scan(sl(p["u"], slice(0, c)), sl(p["delta"], slice(0, c)), p["A"],
                            sl(p["B"], slice(0, c)), sl(p["C"], slice(0, c)),
                            z=sl(p["z"], slice(0, c)), **kw)
    yb, hb, _ = oracle.scan(sl(p["u"], slice(c, None)), sl(p["delta"], slice(c, None)), p["A"],
                            sl(p["B"], slice(c, None)), sl(p["C"], slice(c, None)),
                            z=sl(p["z"], slice(c, None)), h0=ha, **kw)
    np.testing.assert_array_equal(np.concatenate([ya, yb], axis=2), y)
    np.testing.assert_array_equal(hb, hT)


@pytest.mark.parametrize("softplus,zoh", [(True, False), (True, True), (False, True)])
def test_decode_steps_equal_scan(softplus, zoh):
    p = _rand_problem(61, l=30)
    if not softplus:
        p["delta"] = np.abs(p["delta"]) + 0.01
    y, hT, _ = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], dt_bias=p["dt_bias"],
                           D_skip=p["D_skip"], z=p["z"], softplus=softplus, zoh=zoh)
    bt, d, l = p["u"].shape
    state = np.zeros((bt, d, p["A"].shape[1]))
    for t in range(l):
        yt = oracle.state_update(state, p["u"][:, :, t], p["delta"][:, :, t], p["A"],
                                 p["B"][:, :, t], p["C"][:, :, t], dt_bias=p["dt_bias"],
                                 D_skip=p["D_skip"], z=p["z"][:, :, t], softplus=softplus,
                                 zoh=zoh)
        np.testing.assert_array_equal(yt, y[:, :, t])
    np.testing.assert_array_equal(state, hT)


def test_thread_count_independent():
    p = _rand_problem(71, bt=3, d=7, l=33)
    kw = dict(dt_bias=p["dt_bias"], D_skip=p["D_skip"], z=p["z"])
    y1, h1, n1 = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], threads=1, **kw)
    y4, h4, n4 = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], threads=4, **kw)
    assert n1 == 1 and n4 == 4
    np.testing.assert_array_equal(y1, y4)
    np.testing.assert_array_equal(h1, h4)


def test_sampled_rows_match_full():
    shp = synth.ScanShape("t", 2, 24, 4, 50, dtype=synth.BF16, seed=5)
    inp = synth.scan_inputs(shp)
    w = oracle.scan_inputs_f64(inp)
    y, hT, _ = oracle.scan(w["u"], w["delta"], w["A"], w["B"], w["C"], dt_bias=w["dt_bias"],
                           D_skip=w["D_skip"], z=w["z"])
    rows = synth.sample_rows(3, 2, 24, 9)
    ys, hs = oracle.scan_rows(inp, rows)
    np.testing.assert_array_equal(ys, y.reshape(48, 50)[rows])
    np.testing.assert_array_equal(hs, hT.reshape(48, 4)[rows])
