"""Pins for the fp64 oracle's causal depthwise convolution.

* A hand-worked width-3 example with an initial state (tests/golden/conv1d_w3_l4.txt).
* Every row against numpy.convolve (a library routine: full convolution of
  the zero- or state-padded row with the filter reversed in time), with and
  without SiLU, widths 1 to 4.
* Continuation: convolving [0, L1) and then [L1, L) from the first part's
  state equals convolving [0, L) at once.
"""

import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "conv1d_w3_l4.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        vals[k] = np.array([float(x) for x in v])
    return vals


def test_hand_worked_example():
    g = _golden()
    out, st = oracle.conv1d(g["x"][None, None, :], g["weight"][None, :], bias=g["bias"],
                            state=g["state"][None, None, :], silu=False)
    np.testing.assert_allclose(out[0, 0], g["out"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(st[0, 0], g["state_out"], rtol=0, atol=0)


@pytest.mark.parametrize("width", [1, 2, 3, 4])
@pytest.mark.parametrize("silu,with_state", [(False, False), (True, False), (True, True)])
def test_against_numpy_convolve(width, silu, with_state):
    g = np.random.default_rng(width * 7 + silu)
    bt, d, l = 2, 5, 23
    x = g.standard_normal((bt, d, l))
    w = g.standard_normal((d, width))
    bias = g.standard_normal(d)
    state = g.standard_normal((bt, d, width - 1)) if with_state else None
    out, st = oracle.conv1d(x, w, bias=bias, state=state, silu=silu)
    for b in range(bt):
        for c in range(d):
            pad = state[b, c] if with_state else np.zeros(width - 1)
            xp = np.concatenate([pad, x[b, c]])
            full = np.convolve(xp, w[c, ::-1], mode="valid")   # correlation with w
            ref = full + bias[c]
            if silu:
                ref = ref / (1.0 + np.exp(-ref))
            np.testing.assert_allclose(out[b, c], ref, rtol=1e-14, atol=1e-14)
            np.testing.assert_array_equal(st[b, c], xp[len(xp) - (width - 1):])


def test_continuation_through_state():
    g = np.random.default_rng(3)
    x = g.standard_normal((2, 4, 40))
    w = g.standard_normal((4, 4))
    bias = g.standard_normal(4)
    full, st_full = oracle.conv1d(x, w, bias=bias)
    a, st_a = oracle.conv1d(np.ascontiguousarray(x[..., :17]), w, bias=bias)
    b, st_b = oracle.conv1d(np.ascontiguousarray(x[..., 17:]), w, bias=bias, state=st_a)
    np.testing.assert_array_equal(np.concatenate([a, b], axis=2), full)
    np.testing.assert_array_equal(st_b, st_full)
    # a piece shorter than the filter keeps part of the old state
    c, st_c = oracle.conv1d(np.ascontiguousarray(x[..., 17:19]), w, bias=bias, state=st_a)
    np.testing.assert_array_equal(c, full[..., 17:19])
    np.testing.assert_array_equal(st_c, x[..., 16:19])
