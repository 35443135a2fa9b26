"""GPU parity of mamba_scan_bwd (the backward pass) against the fp64 oracle's
reverse-mode gradient, through the C ABI.

Every gradient (du, ddelta, dz, dA, dB, dC, dD_skip, ddt_bias, the initial
state's) is compared element by element on the same seeded inputs: fp32 and
bf16 I/O, dstate 4, 5 and 16, channel counts that leave a partial group of
32 (up to 97 groups), lengths that leave a partial 12-step tile, every
nullable input absent or present, softplus on and off, an initial state and
a final-state gradient.  Most of these shapes have few units of 32 channels,
so the reverse pass runs in time chunks (from 4 up to 67 of them) with the
chunk summaries and their carry.  Tolerances: fp32 I/O max |err| <= 1e-4
max(1, rms(ref)) (fp32 accumulation over the sequence and the channels);
bf16 I/O as the forward (2e-2 of the reference rms, bf16-stored outputs
beyond their own rounding).
"""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, f32_dev, to_dev, to_f64, torch_mod

pytestmark = pytest.mark.gpu


def _inputs(dtype, batch, dim, n, l, seed, softplus=True):
    shp = synth.ScanShape("bwd", batch, dim, n, l, dtype=dtype, softplus=softplus, seed=seed)
    inp = synth.scan_inputs(shp)
    if not softplus:
        mag = np.abs(synth.widen(inp["delta"], dtype)).astype(np.float32) * 0.2 + 0.01
        inp["delta"] = synth.store(mag, dtype)
        inp["dt_bias"] = np.linspace(0.0, 0.05, dim, dtype=np.float32)
    g = np.random.default_rng(seed + 1)
    inp["dy"] = synth.store(g.standard_normal((batch, dim, l)).astype(np.float32), dtype)
    inp["h0"] = (0.5 * g.standard_normal((batch, dim, n))).astype(np.float32)
    inp["dfinal"] = g.standard_normal((batch, dim, n)).astype(np.float32)
    return shp, inp


def _run(inp, z=True, dskip=True, bias=True, h0=False, dfinal=False, softplus=True):
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    dt = inp["dtype"]
    t = lambda k: to_dev(inp[k], dt)
    grads = mm.mamba_scan_bwd(
        t("u"), t("delta"), f32_dev(inp["dt_bias"]) if bias else None, f32_dev(inp["A"]),
        t("B"), t("C"), f32_dev(inp["D_skip"]) if dskip else None, t("z") if z else None,
        t("dy"), softplus=softplus, initial_state=f32_dev(inp["h0"]) if h0 else None,
        d_final_state=f32_dev(inp["dfinal"]) if dfinal else None,
        want_initial_state_grad=True)
    torch.cuda.synchronize()
    w = oracle.scan_inputs_f64(inp)
    ref = oracle.scan_bwd(w["u"], w["delta"], w["A"], w["B"], w["C"],
                          synth.widen(inp["dy"], dt), dt_bias=w["dt_bias"] if bias else None,
                          D_skip=w["D_skip"] if dskip else None, z=w["z"] if z else None,
                          softplus=softplus, h0=inp["h0"] if h0 else None,
                          dfinal=inp["dfinal"] if dfinal else None)
    return grads, ref


PAIRS = [("du", "du"), ("ddelta", "ddelta"), ("dz", "dz"), ("dA", "dA"), ("dB", "dB"),
         ("dC", "dC"), ("dD_skip", "dD"), ("ddt_bias", "ddt_bias"), ("d_initial_state", "dh0")]


def _check(grads, ref, dtype, z=True, dskip=True, bias=True):
    for gk, rk in PAIRS:
        if gk == "dz" and not z:
            assert grads["dz"] is None
            continue
        got = to_f64(grads[gk])
        want = ref[rk]
        if dtype == synth.F32:
            scale = max(1.0, float(np.sqrt(np.mean(want * want))))
            err = float(np.max(np.abs(got - want)))
            assert np.all(np.isfinite(got)) and err <= 1e-4 * scale, (gk, err, scale)
        else:
            stored_bf16 = gk in ("du", "ddelta", "dz")
            assert_close(got, want, dtype, gk, bf16_output=stored_bf16)


SHAPES = [
    # dtype, batch, dim, N, L
    (synth.F32, 1, 16, 4, 64),
    (synth.F32, 2, 33, 5, 70),
    (synth.F32, 1, 40, 16, 129),
    (synth.BF16, 2, 70, 16, 200),
    (synth.BF16, 1, 64, 8, 100),
    (synth.BF16, 2, 128, 16, 1024),
    # 97 groups of 32 channels (the last partial): the dB / dC reduction
    # splits its sum over groups into four parts from 96 groups on
    (synth.BF16, 1, 3104, 16, 100),
    # two units over 4000 steps: the reverse pass in 67 time chunks of five
    # tiles, with the chunk summaries and the carry between them; the same
    # in fp32 over 10 chunks
    (synth.BF16, 1, 64, 16, 4000),
    (synth.F32, 1, 48, 16, 500),
]


@pytest.mark.parametrize("dtype,batch,dim,n,l", SHAPES)
def test_bwd_matches_oracle(dtype, batch, dim, n, l):
    shp, inp = _inputs(dtype, batch, dim, n, l, seed=600 + l + dim)
    grads, ref = _run(inp, h0=True, dfinal=True)
    _check(grads, ref, dtype)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("z,dskip,bias,softplus", [(False, True, True, True),
                                                   (True, False, True, True),
                                                   (True, True, False, True),
                                                   (False, False, False, True),
                                                   (True, True, True, False)])
def test_bwd_nullable_and_softplus(dtype, z, dskip, bias, softplus):
    shp, inp = _inputs(dtype, 2, 70, 16, 150, seed=77, softplus=softplus)
    grads, ref = _run(inp, z=z, dskip=dskip, bias=bias, softplus=softplus)
    _check(grads, ref, dtype, z=z, dskip=dskip, bias=bias)


def test_bwd_chains_through_prefill_pieces():
    # The gradient of a sequence scanned in two pieces (the second from the
    # first's final state) equals the one-piece gradient: run the second
    # piece's backward, feed its d_initial_state to the first piece as
    # d_final_state, and compare with the whole-sequence backward.
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    dtype = synth.F32
    shp, inp = _inputs(dtype, 2, 40, 16, 96, seed=91)
    dt = inp["dtype"]
    cut = 37
    sl = lambda k, s: to_dev(np.ascontiguousarray(inp[k][..., s]), dt)
    A, dtb, dsk = f32_dev(inp["A"]), f32_dev(inp["dt_bias"]), f32_dev(inp["D_skip"])
    full = mm.mamba_scan_bwd(sl("u", slice(None)), sl("delta", slice(None)), dtb, A,
                             sl("B", slice(None)), sl("C", slice(None)), dsk, sl("z", slice(None)),
                             sl("dy", slice(None)))
    # forward of the first piece for the hand-over state
    mid = torch.empty((2, 40, 16), device="cuda")
    mm.mamba_scan_fwd(sl("u", slice(0, cut)), sl("delta", slice(0, cut)), dtb, A,
                      sl("B", slice(0, cut)), sl("C", slice(0, cut)), dsk, sl("z", slice(0, cut)),
                      True, final_state=mid)
    second = mm.mamba_scan_bwd(sl("u", slice(cut, None)), sl("delta", slice(cut, None)), dtb, A,
                               sl("B", slice(cut, None)), sl("C", slice(cut, None)), dsk,
                               sl("z", slice(cut, None)), sl("dy", slice(cut, None)),
                               initial_state=mid, want_initial_state_grad=True)
    first = mm.mamba_scan_bwd(sl("u", slice(0, cut)), sl("delta", slice(0, cut)), dtb, A,
                              sl("B", slice(0, cut)), sl("C", slice(0, cut)), dsk,
                              sl("z", slice(0, cut)), sl("dy", slice(0, cut)),
                              d_final_state=second["d_initial_state"])
    torch.cuda.synchronize()
    for k in ("du", "ddelta", "dz", "dB", "dC"):
        joined = torch.cat([first[k], second[k]], dim=-1)
        err = float((joined - full[k]).abs().max())
        scale = max(1.0, float(full[k].float().pow(2).mean().sqrt()))
        assert err <= 1e-4 * scale, (k, err)
    for k in ("dA", "dD_skip", "ddt_bias"):
        err = float((first[k] + second[k] - full[k]).abs().max())
        scale = max(1.0, float(full[k].pow(2).mean().sqrt()))
        assert err <= 1e-4 * scale, (k, err)


def test_bwd_zero_length():
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    u = torch.empty((2, 8, 0), dtype=torch.bfloat16, device="cuda")
    Bm = torch.empty((2, 4, 0), dtype=torch.bfloat16, device="cuda")
    A = -torch.ones((8, 4), device="cuda")
    dfin = torch.randn((2, 8, 4), device="cuda")
    g = mm.mamba_scan_bwd(u, u.clone(), None, A, Bm, Bm.clone(), None, None, u.clone(),
                          d_final_state=dfin, want_initial_state_grad=True)
    torch.cuda.synchronize()
    assert bool((g["dA"] == 0).all()) and bool((g["d_initial_state"] == dfin).all())


def test_autograd_wrapper_matches_the_backward_call():
    # torch autograd through mamba_scan_fn gives exactly mamba_scan_bwd's
    # gradients (same kernels, same inputs), cast to each input's dtype
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    shp, inp = _inputs(synth.BF16, 2, 70, 16, 150, seed=99)
    dt = inp["dtype"]
    u, delta, z, B, C = (to_dev(inp[k], dt).requires_grad_() for k in ("u", "delta", "z", "B", "C"))
    A, dtb, dsk, h0 = (f32_dev(inp[k]).requires_grad_() for k in ("A", "dt_bias", "D_skip", "h0"))
    dy = to_dev(inp["dy"], dt)
    dfin = f32_dev(inp["dfinal"])
    y, fin = mm.mamba_scan_fn(u, delta, A, B, C, D_skip=dsk, z=z, dt_bias=dtb, initial_state=h0,
                              return_final_state=True)
    ((y.float() * dy.float()).sum() + (fin * dfin).sum()).backward()
    g = mm.mamba_scan_bwd(u.detach(), delta.detach(), dtb.detach(), A.detach(), B.detach(),
                          C.detach(), dsk.detach(), z.detach(), dy, initial_state=h0.detach(),
                          d_final_state=dfin, want_initial_state_grad=True)
    y2 = mm.mamba_scan_fwd_ex(u.detach(), delta.detach(), dtb.detach(), A.detach(), B.detach(),
                              C.detach(), dsk.detach(), z.detach(), initial_state=h0.detach())
    torch.cuda.synchronize()
    assert torch.equal(y.detach(), y2)
    for t, k in ((u, "du"), (delta, "ddelta"), (z, "dz"), (A, "dA"), (dtb, "ddt_bias"),
                 (dsk, "dD_skip"), (h0, "d_initial_state")):
        assert torch.equal(t.grad, g[k].to(t.dtype)), k
    for t, k in ((B, "dB"), (C, "dC")):
        assert torch.equal(t.grad, g[k].to(t.dtype)), k
    # without the final state only y is returned and differentiable
    u.grad = None
    y3 = mm.mamba_scan_fn(u, delta, A, B, C, D_skip=dsk, z=z, dt_bias=dtb)
    (y3.float() * dy.float()).sum().backward()
    g3 = mm.mamba_scan_bwd(u.detach(), delta.detach(), dtb.detach(), A.detach(), B.detach(),
                           C.detach(), dsk.detach(), z.detach(), dy)
    torch.cuda.synchronize()
    assert torch.equal(u.grad, g3["du"])


@pytest.mark.slow
def test_bwd_fills_the_gpu_bf16():
    """bf16, batch 2 x 1536 channels x N 16 x 2048 steps: 96 groups of 32
    channels, more than one per SM, so the dB / dC reductions over the
    channels add many per-warp partials.  Every gradient, with an initial
    state and a final-state gradient, element by element against the oracle."""
    shp, inp = _inputs(synth.BF16, 2, 1536, 16, 2048, seed=61)
    grads, ref = _run(inp, h0=True, dfinal=True)
    _check(grads, ref, synth.BF16)
    import selective_state_space_135_b300 as mm
    assert mm.mamba_device_status() == 0
