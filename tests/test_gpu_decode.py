"""GPU parity of mamba_state_update (generation step) against the fp64 oracle,
and decode == scan: 1024 single-token steps from a zero state must agree with
one mamba_scan_fwd over the same 1024 tokens."""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, f32_dev, to_dev, to_f64, torch_mod

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,batch,dim,n,zgate", [
    (synth.F32, 3, 37, 16, True), (synth.F32, 2, 5, 1, False), (synth.F32, 1, 64, 5, True),
    (synth.BF16, 4, 130, 16, True), (synth.BF16, 2, 33, 13, False), (synth.BF16, 1, 8, 4, True),
    # dstate 16 over two blocks of 8 batch entries, the second with one
    (synth.BF16, 9, 70, 16, True),
])
def test_decode_small(dtype, batch, dim, n, zgate):
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    shp = synth.DecodeShape("small", batch, dim, n, 6, dtype=dtype, seed=31 + dim)
    par = synth.decode_params(shp)
    g = np.random.default_rng(3)
    h0 = g.standard_normal((batch, dim, n)) * 0.3
    state = f32_dev(h0)
    href = h0.astype(np.float32).astype(np.float64)
    for step in range(shp.steps):
        si = synth.decode_step_inputs(shp, step)
        y = mm.mamba_state_update(state, to_dev(si["x"], dtype), to_dev(si["delta"], dtype),
                                  f32_dev(par["dt_bias"]), f32_dev(par["A"]),
                                  to_dev(si["B"], dtype), to_dev(si["C"], dtype),
                                  f32_dev(par["D_skip"]),
                                  to_dev(si["z"], dtype) if zgate else None)
        yr = oracle.state_update(href, synth.widen(si["x"], dtype), synth.widen(si["delta"], dtype),
                                 par["A"], synth.widen(si["B"], dtype), synth.widen(si["C"], dtype),
                                 dt_bias=par["dt_bias"], D_skip=par["D_skip"],
                                 z=synth.widen(si["z"], dtype) if zgate else None)
        torch.cuda.synchronize()
        assert_close(to_f64(y), yr, dtype, f"y step {step}")
    assert_close(to_f64(state), href, dtype, "state")


@pytest.mark.slow
def test_decode_workload_matches_oracle_and_scan():
    """The batched decode workload: (128, 5120, 16) fp32 state, 1024 steps."""
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    shp = synth.DECODE
    bt, d, n, steps = shp.batch, shp.dim, shp.dstate, shp.steps
    par = synth.decode_params(shp)
    A, dtb, dsk = f32_dev(par["A"]), f32_dev(par["dt_bias"]), f32_dev(par["D_skip"])
    state = torch.zeros((bt, d, n), device="cuda")
    # sampled sub-grid for the oracle: 8 batch entries x 32 channels
    gs = np.random.default_rng(4)
    bs = np.sort(gs.choice(bt, 8, replace=False))
    ds = np.sort(gs.choice(d, 32, replace=False))
    href = np.zeros((len(bs), len(ds), n))
    bs_t = torch.as_tensor(bs, device="cuda")
    ds_t = torch.as_tensor(ds, device="cuda")
    # full per-step inputs stacked on the device for the scan comparison
    bf = torch.bfloat16
    U = torch.empty((bt, d, steps), dtype=bf, device="cuda")
    DL = torch.empty_like(U)
    Z = torch.empty_like(U)
    Bs = torch.empty((bt, n, steps), dtype=bf, device="cuda")
    Cs = torch.empty_like(Bs)
    Yd = torch.empty((bt, d, steps), dtype=bf, device="cuda")
    ysub_gpu, ysub_ref = [], []
    for step in range(steps):
        si = synth.decode_step_inputs(shp, step)
        x, dl, z = (to_dev(si[k], shp.dtype) for k in ("x", "delta", "z"))
        Bt, Ct = to_dev(si["B"], shp.dtype), to_dev(si["C"], shp.dtype)
        y = mm.mamba_state_update(state, x, dl, dtb, A, Bt, Ct, dsk, z)
        U[:, :, step] = x
        DL[:, :, step] = dl
        Z[:, :, step] = z
        Bs[:, :, step] = Bt
        Cs[:, :, step] = Ct
        Yd[:, :, step] = y
        sub = lambda a: synth.widen(a[np.ix_(bs, ds)], shp.dtype)
        yr = oracle.state_update(href, sub(si["x"]), sub(si["delta"]), par["A"][ds],
                                 synth.widen(si["B"][bs], shp.dtype),
                                 synth.widen(si["C"][bs], shp.dtype),
                                 dt_bias=par["dt_bias"][ds], D_skip=par["D_skip"][ds],
                                 z=sub(si["z"]))
        ysub_ref.append(yr)
        ysub_gpu.append(y.index_select(0, bs_t).index_select(1, ds_t))
    torch.cuda.synchronize()
    yg = np.stack([to_f64(t) for t in ysub_gpu])
    st = assert_close(yg, np.stack(ysub_ref), shp.dtype, "decode y (sampled)")
    sg = to_f64(state.index_select(0, bs_t).index_select(1, ds_t))
    assert_close(sg, href, shp.dtype, "decode state (sampled)")
    # decode == scan over the same tokens, on the whole state
    fin = torch.empty((bt, d, n), device="cuda")
    Ys = mm.mamba_scan_fwd(U, DL, dtb, A, Bs, Cs, dsk, Z, True, final_state=fin)
    torch.cuda.synchronize()
    # both sides are bf16-rounded fp32 results: allow one bf16 round-off each
    ysf, ydf = Ys.float(), Yd.float()
    rms = ydf.pow(2).mean().sqrt().item()
    excess = ((ysf - ydf).abs() - 2.0 * 2.0 ** -8 * ydf.abs()).max().item()
    diff = (ysf - ydf).pow(2).mean().sqrt().item()
    assert diff / rms <= 2e-2, (diff, rms)
    assert excess / rms <= 2e-2, (excess, rms)
    sd = (fin - state).abs().max().item()
    srms = state.pow(2).mean().sqrt().item()
    assert sd / srms <= 2e-2, (sd, srms)
    print("decode", st, "scan-vs-decode", diff / rms, sd / srms)
