"""Pins for the fp64 oracle's backward pass (reverse-mode gradient of the
scan), against the forward oracle, which test_oracle_pins.py pins in turn.

* Central finite differences of J = sum(dy * y) + sum(dfinal * final_state)
  for every element of every input (u, delta, z, B, C, A, D_skip, dt_bias,
  the initial state), with softplus, gate, skip, bias, initial state and
  final-state gradient on, and with all of them off.
* Exact adjoint identities where the forward is linear: y in u (zero
  initial state), (y, final state) in the initial state (u = 0), y in C.

A dropped term, a wrong sign or index, or a gradient routed to the wrong
input fails the finite differences at a few 1e-7 of relative error.
"""

import numpy as np
import pytest

import oracle


def _problem(seed, bt=2, d=3, n=4, l=10, full=True):
    g = np.random.default_rng(seed)
    p = dict(
        u=g.standard_normal((bt, d, l)),
        delta=0.5 * g.standard_normal((bt, d, l)) if full else np.abs(g.standard_normal((bt, d, l))) * 0.3 + 0.05,
        A=-g.uniform(0.3, 3.0, (d, n)),
        B=g.standard_normal((bt, n, l)),
        C=g.standard_normal((bt, n, l)),
        dt_bias=g.uniform(-2.0, 0.5, d) if full else None,
        D_skip=g.standard_normal(d) if full else None,
        z=g.standard_normal((bt, d, l)) if full else None,
        h0=0.5 * g.standard_normal((bt, d, n)) if full else None,
    )
    dy = g.standard_normal((bt, d, l))
    dfinal = g.standard_normal((bt, d, n)) if full else None
    return p, dy, dfinal


def _loss(p, dy, dfinal, softplus):
    y, hT, _ = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], dt_bias=p["dt_bias"],
                           D_skip=p["D_skip"], z=p["z"], softplus=softplus, h0=p["h0"])
    j = float(np.sum(dy * y))
    if dfinal is not None:
        j += float(np.sum(dfinal * hT))
    return j


GRAD_OF = {"u": "du", "delta": "ddelta", "z": "dz", "B": "dB", "C": "dC", "A": "dA",
           "D_skip": "dD", "dt_bias": "ddt_bias", "h0": "dh0"}


@pytest.mark.parametrize("full,softplus", [(True, True), (False, False), (True, False)])
def test_gradients_match_central_differences(full, softplus):
    p, dy, dfinal = _problem(3 if full else 4, full=full)
    if full and not softplus:
        p["delta"] = np.abs(p["delta"]) * 0.3 + 0.05      # Delta = delta + dt_bias stays > 0
        p["dt_bias"] = np.abs(p["dt_bias"]) * 0.1
    grads = oracle.scan_bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], dy,
                            dt_bias=p["dt_bias"], D_skip=p["D_skip"], z=p["z"],
                            softplus=softplus, h0=p["h0"], dfinal=dfinal)
    checked = 0
    for name, gname in GRAD_OF.items():
        if p[name] is None:
            continue
        x = p[name]
        gx = grads[gname]
        assert gx is not None and gx.shape == x.shape, name
        for idx in np.ndindex(x.shape):
            old = x[idx]
            eps = 1e-6 * max(1.0, abs(old))
            x[idx] = old + eps
            jp = _loss(p, dy, dfinal, softplus)
            x[idx] = old - eps
            jm = _loss(p, dy, dfinal, softplus)
            x[idx] = old
            fd = (jp - jm) / (2 * eps)
            assert abs(fd - gx[idx]) <= 2e-7 * max(1.0, abs(fd)), (name, idx, fd, gx[idx])
            checked += 1
    assert checked == sum(p[k].size for k in GRAD_OF if p[k] is not None)


def test_adjoint_identity_in_u():
    # h0 = 0, no gate: y = M u exactly, so <dy, y(v)> = <du(dy), v>
    p, dy, _ = _problem(5)
    p["z"] = None
    p["h0"] = None
    grads = oracle.scan_bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], dy,
                            dt_bias=p["dt_bias"], D_skip=p["D_skip"])
    v = np.random.default_rng(6).standard_normal(p["u"].shape)
    y, _, _ = oracle.scan(v, p["delta"], p["A"], p["B"], p["C"], dt_bias=p["dt_bias"],
                          D_skip=p["D_skip"])
    lhs, rhs = float(np.sum(dy * y)), float(np.sum(grads["du"] * v))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_adjoint_identity_in_initial_state():
    # u = 0, no gate: (y, final state) are linear in h0
    p, dy, dfinal = _problem(7)
    p["z"] = None
    p["u"] = np.zeros_like(p["u"])
    grads = oracle.scan_bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], dy,
                            dt_bias=p["dt_bias"], D_skip=p["D_skip"], h0=p["h0"], dfinal=dfinal)
    v = np.random.default_rng(8).standard_normal(p["h0"].shape)
    y, hT, _ = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], dt_bias=p["dt_bias"],
                           D_skip=p["D_skip"], h0=v)
    lhs = float(np.sum(dy * y) + np.sum(dfinal * hT))
    rhs = float(np.sum(grads["dh0"] * v))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_adjoint_identity_in_C():
    # y is affine in C: <dy, y(C + V) - y(C)> = <dC, V>
    p, dy, _ = _problem(9)
    p["z"] = None
    grads = oracle.scan_bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], dy,
                            dt_bias=p["dt_bias"], D_skip=p["D_skip"], h0=p["h0"])
    V = np.random.default_rng(10).standard_normal(p["C"].shape)
    kw = dict(dt_bias=p["dt_bias"], D_skip=p["D_skip"], h0=p["h0"])
    y0, _, _ = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], **kw)
    y1, _, _ = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"] + V, **kw)
    lhs, rhs = float(np.sum(dy * (y1 - y0))), float(np.sum(grads["dC"] * V))
    assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs))
