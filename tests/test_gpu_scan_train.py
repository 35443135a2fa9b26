"""GPU checks of the training pair mamba_scan_fwd_train / mamba_scan_bwd_ckpt.

* The training forward's y and final state are bit for bit those of
  mamba_scan_fwd_ex on the same inputs and initial state (same kernels and
  plan; it only also stores the state every 12 steps).
* Its checkpoints hold the state before steps 0, 12, 24, ...: checkpoint 0
  is the initial state exactly, and every later one is compared with the
  fp64 oracle's state after the same prefix of the sequence.
* mamba_scan_bwd_ckpt from those checkpoints gives, bit for bit, the
  gradients of mamba_scan_bwd, which recomputes the checkpoints itself (the
  parity of those gradients with the oracle is tested in
  test_gpu_scan_bwd.py); whole-sequence and time-chunked plans.
* mamba_scan_fn with keep_checkpoints runs through this pair with the same
  results.
"""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, f32_dev, to_dev, to_f64, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_tuning():
    import selective_state_space_135_b300 as mm
    mm.mamba_scan_set_tuning(0, 0, 0, 0)
    yield
    mm.mamba_scan_set_tuning(0, 0, 0, 0)


def _inputs(dtype, batch, dim, n, l, seed):
    shp = synth.ScanShape("train", batch, dim, n, l, dtype=dtype, seed=seed)
    inp = synth.scan_inputs(shp)
    g = np.random.default_rng(seed + 1)
    inp["dy"] = synth.store(g.standard_normal((batch, dim, l)).astype(np.float32), dtype)
    inp["h0"] = (0.5 * g.standard_normal((batch, dim, n))).astype(np.float32)
    inp["dfinal"] = g.standard_normal((batch, dim, n)).astype(np.float32)
    return inp


def _dev(inp, z=True):
    dt = inp["dtype"]
    return (to_dev(inp["u"], dt), to_dev(inp["delta"], dt), f32_dev(inp["dt_bias"]),
            f32_dev(inp["A"]), to_dev(inp["B"], dt), to_dev(inp["C"], dt),
            f32_dev(inp["D_skip"]), to_dev(inp["z"], dt) if z else None)


CASES = [
    # dtype, batch, dim, N, L, time chunks (0: the planner's choice), initial state, z
    (synth.F32, 1, 40, 16, 129, 0, True, True),
    (synth.F32, 2, 33, 5, 70, 0, False, False),
    (synth.BF16, 2, 70, 16, 200, 0, True, True),
    (synth.BF16, 1, 64, 8, 100, 0, False, True),
    (synth.BF16, 2, 128, 16, 1024, 3, True, True),
    (synth.BF16, 1, 96, 4, 600, 4, False, True),
]


@pytest.mark.parametrize("dtype,batch,dim,n,l,chunks,h0,z", CASES)
def test_train_pair_matches_the_plain_calls(dtype, batch, dim, n, l, chunks, h0, z):
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    inp = _inputs(dtype, batch, dim, n, l, seed=700 + l + dim)
    args = _dev(inp, z)
    h0t = f32_dev(inp["h0"]) if h0 else None
    dy = to_dev(inp["dy"], dtype)
    dfin = f32_dev(inp["dfinal"])
    mm.mamba_scan_set_tuning(0, 0, chunks)
    fin_t = torch.empty((batch, dim, n), device="cuda")
    y_t, ck = mm.mamba_scan_fwd_train(*args, softplus=True, initial_state=h0t, final_state=fin_t)
    fin_e = torch.empty((batch, dim, n), device="cuda")
    y_e = mm.mamba_scan_fwd_ex(*args, softplus=True, initial_state=h0t, final_state=fin_e)
    g_ck = mm.mamba_scan_bwd_ckpt(*args, dy, ck, softplus=True, d_final_state=dfin,
                                  want_initial_state_grad=True)
    g = mm.mamba_scan_bwd(*args, dy, softplus=True, initial_state=h0t, d_final_state=dfin,
                          want_initial_state_grad=True)
    torch.cuda.synchronize()
    assert mm.mamba_device_status() == 0
    assert torch.equal(y_t, y_e)
    assert torch.equal(fin_t, fin_e)
    for k, v in g.items():
        if v is None:
            assert g_ck[k] is None, k
        else:
            assert torch.equal(g_ck[k], v), k
    # the checkpoints: shape, zero padding of the state, the initial state at
    # k = 0, the oracle's state after 12 k steps for a few later k
    assert tuple(ck.shape) == mm.checkpoint_shape(batch, dim, n, l)
    # (batch, tile, quad, dim, 4) -> (batch, tile, dim, padded state)
    c = ck.permute(0, 1, 3, 2, 4).reshape(batch, ck.shape[1], dim, -1).cpu().numpy()
    c = c.astype(np.float64)
    assert np.all(c[..., n:] == 0.0)
    want0 = inp["h0"] if h0 else np.zeros((batch, dim, n), np.float32)
    assert np.array_equal(c[:, 0, :, :n], want0.astype(np.float64))
    w = oracle.scan_inputs_f64(inp)
    for k in sorted({1, ck.shape[1] // 2, ck.shape[1] - 1}):
        if k == 0:
            continue
        s = 12 * k
        sub = lambda a: None if a is None else np.ascontiguousarray(a[..., :s])
        _, hk, _ = oracle.scan(sub(w["u"]), sub(w["delta"]), w["A"], sub(w["B"]), sub(w["C"]),
                               dt_bias=w["dt_bias"], D_skip=None, z=None, softplus=True,
                               h0=inp["h0"] if h0 else None)
        assert_close(c[:, k, :, :n], hk, dtype, f"checkpoint {k}")


def test_autograd_keep_checkpoints_matches():
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    inp = _inputs(synth.BF16, 2, 70, 16, 150, seed=99)
    dt = inp["dtype"]
    grads = []
    for keep in (False, True):
        u, delta, z, B, C = (to_dev(inp[k], dt).requires_grad_()
                             for k in ("u", "delta", "z", "B", "C"))
        A, dtb, dsk, h0 = (f32_dev(inp[k]).requires_grad_()
                           for k in ("A", "dt_bias", "D_skip", "h0"))
        dy = to_dev(inp["dy"], dt)
        y = mm.mamba_scan_fn(u, delta, A, B, C, D_skip=dsk, z=z, dt_bias=dtb, initial_state=h0,
                             keep_checkpoints=keep)
        (y.float() * dy.float()).sum().backward()
        grads.append([y.detach()] + [t.grad for t in (u, delta, z, B, C, A, dtb, dsk, h0)])
    torch.cuda.synchronize()
    for a, b in zip(*grads):
        assert torch.equal(a, b)


def test_train_pair_zero_length():
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    u = torch.empty((2, 8, 0), dtype=torch.bfloat16, device="cuda")
    Bm = torch.empty((2, 4, 0), dtype=torch.bfloat16, device="cuda")
    A = -torch.ones((8, 4), device="cuda")
    h0 = torch.randn((2, 8, 4), device="cuda")
    fin = torch.empty((2, 8, 4), device="cuda")
    y, ck = mm.mamba_scan_fwd_train(u, u.clone(), None, A, Bm, Bm.clone(), None, None,
                                    initial_state=h0, final_state=fin)
    dfin = torch.randn((2, 8, 4), device="cuda")
    g = mm.mamba_scan_bwd_ckpt(u, u.clone(), None, A, Bm, Bm.clone(), None, None, u.clone(), ck,
                               d_final_state=dfin, want_initial_state_grad=True)
    torch.cuda.synchronize()
    assert ck.numel() == 0 and torch.equal(fin, h0)
    assert bool((g["dA"] == 0).all()) and torch.equal(g["d_initial_state"], dfin)


@pytest.mark.slow
def test_train_pair_bitwise_on_the_130m_layer():
    """The Mamba-130M layer workload (B8 D1536 N16 L2048 bf16, 384 units of 32
    channels, the backward's full wave): the training pair against the plain
    calls, bit for bit, every output and gradient."""
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    inp = synth.scan_inputs(synth.M130)
    args = _dev(inp)
    g = torch.Generator(device="cuda").manual_seed(5)
    dy = torch.randn(args[0].shape, device="cuda", generator=g).to(args[0].dtype)
    dfin = torch.randn((8, 1536, 16), device="cuda", generator=g)
    fin_t = torch.empty((8, 1536, 16), device="cuda")
    fin = torch.empty_like(fin_t)
    y_t, ck = mm.mamba_scan_fwd_train(*args, final_state=fin_t)
    y = mm.mamba_scan_fwd(*args, final_state=fin)
    g_ck = mm.mamba_scan_bwd_ckpt(*args, dy, ck, d_final_state=dfin, want_initial_state_grad=True)
    g_pl = mm.mamba_scan_bwd(*args, dy, d_final_state=dfin, want_initial_state_grad=True)
    torch.cuda.synchronize()
    assert mm.mamba_device_status() == 0
    assert torch.equal(y_t, y) and torch.equal(fin_t, fin)
    for k, v in g_pl.items():
        assert torch.equal(g_ck[k], v), k
