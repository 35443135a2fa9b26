"""fp64 CPU oracle for the selective scan (S6) and its decode state update.

TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg use this module.  The CUDA library neither
imports nor links it, and the two share no code; inputs reach both from the
seeded generators in ``synth``.

The arithmetic lives in ``oracle_scan.c`` (plain C, fp64, one (b, d) row at
a time, time-sequential).  This file only builds it with gcc, widens inputs
to float64 and marshals pointers.  See the C file's header for the formula
and the page it follows.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
closed forms and independent formulations (Theorem 1's gated RNN, the
keep/reset limits, the explicitly unrolled sum, the time-invariant
convolution, linearity, causality); the backward pass ``scan_bwd`` by
``tests/test_oracle_bwd_pins.py`` (central finite differences of the
forward for every input, and exact adjoint identities); the causal
convolution ``conv1d`` by ``tests/test_oracle_conv_pins.py``
(numpy.convolve, a hand-worked example, continuation through the state).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_scan.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_scan.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc into oracle/liboracle_scan.so."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.oracle_scan_f64.argtypes = [i64, i64, i64, i64, P, P, P, P, P, P, P, P,
                                            ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_int]
            lib.oracle_scan_f64.restype = ctypes.c_int
            lib.oracle_state_update_f64.argtypes = [i64, i64, i64, P, P, P, P, P, P, P, P, P,
                                                    ctypes.c_int, ctypes.c_int, P]
            lib.oracle_state_update_f64.restype = ctypes.c_int
            lib.oracle_scan_bwd_f64.argtypes = [i64, i64, i64, i64] + [P] * 8 + [ctypes.c_int] \
                + [P] * 12
            lib.oracle_scan_bwd_f64.restype = ctypes.c_int
            lib.oracle_conv1d_f64.argtypes = [i64, i64, i64, i64, P, P, P, P, ctypes.c_int, P, P]
            lib.oracle_conv1d_f64.restype = ctypes.c_int
            lib.oracle_softplus_f64.argtypes = [ctypes.c_double]
            lib.oracle_softplus_f64.restype = ctypes.c_double
            lib.oracle_zoh_weight_f64.argtypes = [ctypes.c_double, ctypes.c_double]
            lib.oracle_zoh_weight_f64.restype = ctypes.c_double
            lib.oracle_silu_f64.argtypes = [ctypes.c_double]
            lib.oracle_silu_f64.restype = ctypes.c_double
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def softplus(s: float) -> float:
    return _load().oracle_softplus_f64(float(s))


def silu(z: float) -> float:
    return _load().oracle_silu_f64(float(z))


def zoh_weight(dt: float, a: float) -> float:
    return _load().oracle_zoh_weight_f64(float(dt), float(a))


def scan(u, delta, A, B, C, dt_bias=None, D_skip=None, z=None, softplus: bool = True,
         h0=None, threads: Optional[int] = None, zoh: bool = False
         ) -> Tuple[np.ndarray, np.ndarray, int]:
    """Selective scan in fp64.

    u, delta, z: (batch, D, L); B, C: (batch, N, L); A: (D, N);
    dt_bias, D_skip: (D,); h0: optional (batch, D, N) initial state; zoh
    selects the zero-order-hold input term instead of Euler's.
    Returns (y (batch, D, L), final state (batch, D, N), threads used).
    """
    u, delta, A, B, C = map(_f64, (u, delta, A, B, C))
    dt_bias, D_skip, z, h0 = map(_f64, (dt_bias, D_skip, z, h0))
    bt, d, l = u.shape
    n = A.shape[1]
    assert delta.shape == u.shape and B.shape == (bt, n, l) and C.shape == (bt, n, l)
    assert A.shape == (d, n)
    if z is not None:
        assert z.shape == u.shape
    if h0 is not None:
        assert h0.shape == (bt, d, n)
    y = np.empty((bt, d, l), dtype=np.float64)
    hT = np.empty((bt, d, n), dtype=np.float64)
    rc = _load().oracle_scan_f64(bt, d, n, l, _ptr(u), _ptr(delta), _ptr(dt_bias), _ptr(A),
                                 _ptr(B), _ptr(C), _ptr(D_skip), _ptr(z), int(bool(softplus)),
                                 int(bool(zoh)), _ptr(h0), _ptr(y), _ptr(hT), int(threads or 0))
    if rc <= 0:
        raise RuntimeError(f"oracle_scan_f64 failed: {rc}")
    return y, hT, rc


def scan_bwd(u, delta, A, B, C, dy, dt_bias=None, D_skip=None, z=None, softplus: bool = True,
             h0=None, dfinal=None) -> dict:
    """Gradients of J = sum(dy * y) + sum(dfinal * final_state) with respect
    to every input of ``scan`` (Euler input term), in fp64.  Returns a dict
    with du, ddelta, dz (or None), dA, dB, dC, dD, ddt_bias and dh0."""
    u, delta, A, B, C, dy = map(_f64, (u, delta, A, B, C, dy))
    dt_bias, D_skip, z, h0, dfinal = map(_f64, (dt_bias, D_skip, z, h0, dfinal))
    bt, d, l = u.shape
    n = A.shape[1]
    assert dy.shape == u.shape and B.shape == (bt, n, l) and C.shape == (bt, n, l)
    out = dict(du=np.empty((bt, d, l)), ddelta=np.empty((bt, d, l)),
               dz=None if z is None else np.empty((bt, d, l)), dA=np.empty((d, n)),
               dB=np.empty((bt, n, l)), dC=np.empty((bt, n, l)), dD=np.empty(d),
               ddt_bias=np.empty(d), dh0=np.empty((bt, d, n)))
    rc = _load().oracle_scan_bwd_f64(
        bt, d, n, l, _ptr(u), _ptr(delta), _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C),
        _ptr(D_skip), _ptr(z), int(bool(softplus)), _ptr(h0), _ptr(dy), _ptr(dfinal),
        _ptr(out["du"]), _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]),
        _ptr(out["dD"]), _ptr(out["dz"]), _ptr(out["ddt_bias"]), _ptr(out["dh0"]))
    if rc != 0:
        raise RuntimeError(f"oracle_scan_bwd_f64 failed: {rc}")
    return out


def conv1d(x, weight, bias=None, state=None, silu: bool = True):
    """Causal depthwise convolution (width W = weight.shape[1]) with an
    optional SiLU, in fp64.  x: (batch, D, L); weight: (D, W); bias: (D,);
    state: optional (batch, D, W - 1), the inputs before t = 0, oldest first.
    Returns (out (batch, D, L), state after the last input (batch, D, W - 1))."""
    x, weight, bias, state = map(_f64, (x, weight, bias, state))
    bt, d, l = x.shape
    w = weight.shape[1]
    assert weight.shape == (d, w)
    if state is not None:
        assert state.shape == (bt, d, w - 1)
    out = np.empty((bt, d, l))
    st = np.empty((bt, d, w - 1))
    rc = _load().oracle_conv1d_f64(bt, d, l, w, _ptr(x), _ptr(weight), _ptr(bias), _ptr(state),
                                   int(bool(silu)), _ptr(out), _ptr(st))
    if rc != 0:
        raise RuntimeError(f"oracle_conv1d_f64 failed: {rc}")
    return out, st


def state_update(state, x, delta, A, B, C, dt_bias=None, D_skip=None, z=None,
                 softplus: bool = True, zoh: bool = False):
    """One decode step in fp64, in place on ``state`` (batch, D, N) float64.

    x, delta, z: (batch, D); B, C: (batch, N).  Returns y (batch, D).
    """
    assert state.dtype == np.float64 and state.flags.c_contiguous
    x, delta, A, B, C = map(_f64, (x, delta, A, B, C))
    dt_bias, D_skip, z = map(_f64, (dt_bias, D_skip, z))
    bt, d, n = state.shape
    y = np.empty((bt, d), dtype=np.float64)
    rc = _load().oracle_state_update_f64(bt, d, n, _ptr(state), _ptr(x), _ptr(delta),
                                         _ptr(dt_bias), _ptr(A), _ptr(B), _ptr(C),
                                         _ptr(D_skip), _ptr(z), int(bool(softplus)),
                                         int(bool(zoh)), _ptr(y))
    if rc != 0:
        raise RuntimeError(f"oracle_state_update_f64 failed: {rc}")
    return y


def scan_inputs_f64(inp: dict, rows=None):
    """Widen a ``synth.scan_inputs`` dict to float64 oracle arguments.

    With ``rows`` (flat b*D + d indices) the result is a smaller problem with
    one batch entry per row (batch = len(rows), D = 1), each carrying its own
    copy of B and C for its batch, so long workloads can be checked on a
    sample of rows.
    """
    import synth
    dt = inp["dtype"]
    A = np.asarray(inp["A"], dtype=np.float64)
    dtb = np.asarray(inp["dt_bias"], dtype=np.float64)
    dsk = np.asarray(inp["D_skip"], dtype=np.float64)
    zs = inp.get("z")
    if rows is None:
        return dict(u=synth.widen(inp["u"], dt), delta=synth.widen(inp["delta"], dt),
                    z=None if zs is None else synth.widen(zs, dt),
                    B=synth.widen(inp["B"], dt), C=synth.widen(inp["C"], dt),
                    A=A, dt_bias=dtb, D_skip=dsk)
    d = inp["u"].shape[1]
    rows = np.asarray(rows, dtype=np.int64)
    bi, di = rows // d, rows % d
    # slice in storage form first, then widen only the sampled rows
    out = dict(u=synth.widen(inp["u"][bi, di], dt)[:, None, :],
               delta=synth.widen(inp["delta"][bi, di], dt)[:, None, :],
               z=None if zs is None else synth.widen(zs[bi, di], dt)[:, None, :],
               B=synth.widen(inp["B"][bi], dt), C=synth.widen(inp["C"][bi], dt))
    # with D = 1 every "batch" entry is one original row, so A/dt_bias/D_skip
    # are per row; scan_rows runs one problem per distinct channel d.
    out.update(A=A[di], dt_bias=dtb[di], D_skip=dsk[di], rows_d=di)
    return out


def scan_rows(inp: dict, rows, threads: Optional[int] = None):
    """Oracle y (len(rows), L) and final state (len(rows), N) for sampled rows."""
    w = scan_inputs_f64(inp, rows)
    R = len(rows)
    L = w["u"].shape[2]
    N = w["A"].shape[1]
    ys = np.empty((R, L))
    hs = np.empty((R, N))
    # group rows by channel d so each oracle call has one A/dt_bias/D_skip row
    order = np.argsort(w["rows_d"], kind="stable")
    di_sorted = w["rows_d"][order]
    starts = np.flatnonzero(np.r_[True, di_sorted[1:] != di_sorted[:-1]])
    ends = np.r_[starts[1:], len(order)]
    for s, e in zip(starts, ends):
        idx = order[s:e]
        y, hT, _ = scan(w["u"][idx], w["delta"][idx], w["A"][idx[:1]], w["B"][idx],
                        w["C"][idx], dt_bias=w["dt_bias"][idx[:1]],
                        D_skip=w["D_skip"][idx[:1]],
                        z=None if w["z"] is None else w["z"][idx],
                        softplus=inp.get("softplus", True), threads=threads)
        ys[idx] = y[:, 0, :]
        hs[idx] = hT[:, 0, :]
    return ys, hs
