"""GPU parity of the causal convolution (mamba_conv1d_fwd, mamba_conv1d_update)
against the fp64 oracle, through the C ABI: fp32 and bf16, widths 1 to 8,
with and without SiLU, bias and a carried state, lengths with a ragged
last run of 8; the carried-out state is compared bit for bit (it is a copy
of inputs), a sequence cut into pieces chained through the state matches
the whole, and generation steps reproduce the sequence kernel bit for bit.
"""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, f32_dev, to_dev, to_f64, torch_mod

pytestmark = pytest.mark.gpu


def _inputs(dtype, batch, dim, l, width, seed):
    g = np.random.default_rng(seed)
    x = synth.store(g.standard_normal((batch, dim, l)).astype(np.float32), dtype)
    w = (g.standard_normal((dim, width)) / np.sqrt(width)).astype(np.float32)
    bias = g.standard_normal(dim).astype(np.float32)
    state = synth.store(g.standard_normal((batch, dim, width - 1)).astype(np.float32), dtype)
    return x, w, bias, state


CASES = [
    # dtype, batch, dim, L, width
    (synth.F32, 1, 5, 1, 4),
    (synth.F32, 2, 33, 63, 4),
    (synth.F32, 1, 16, 1000, 3),
    (synth.F32, 2, 7, 40, 1),
    (synth.BF16, 1, 5, 7, 4),
    (synth.BF16, 2, 130, 1000, 4),
    (synth.BF16, 3, 64, 2048, 2),
    (synth.BF16, 1, 40, 129, 8),
]


@pytest.mark.parametrize("dtype,batch,dim,l,width", CASES)
@pytest.mark.parametrize("silu,with_state,with_bias", [(True, True, True), (False, False, True),
                                                       (True, False, False)])
def test_conv_matches_oracle(dtype, batch, dim, l, width, silu, with_state, with_bias):
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    x, w, bias, state = _inputs(dtype, batch, dim, l, width, seed=l + 13 * width + dim)
    fin = torch.empty((batch, dim, width - 1), dtype=torch.float32 if dtype == synth.F32
                      else torch.bfloat16, device="cuda")
    out = mm.mamba_conv1d_fwd(to_dev(x, dtype), f32_dev(w), f32_dev(bias) if with_bias else None,
                              to_dev(state, dtype) if with_state else None, silu=silu,
                              final_conv_state=fin)
    torch.cuda.synchronize()
    ref, ref_state = oracle.conv1d(synth.widen(x, dtype), w, bias=bias if with_bias else None,
                                   state=synth.widen(state, dtype) if with_state else None,
                                   silu=silu)
    assert_close(to_f64(out), ref, dtype, "conv out")
    np.testing.assert_array_equal(to_f64(fin), ref_state)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_conv_pieces_chain_through_the_state(dtype):
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    x, w, bias, _ = _inputs(dtype, 2, 70, 300, 4, seed=5)
    xd, wd, bd = to_dev(x, dtype), f32_dev(w), f32_dev(bias)
    full = mm.mamba_conv1d_fwd(xd, wd, bd)
    tdt = xd.dtype
    s1 = torch.empty((2, 70, 3), dtype=tdt, device="cuda")
    s2 = torch.empty_like(s1)
    s3 = torch.empty_like(s1)
    a = mm.mamba_conv1d_fwd(xd[..., :101].contiguous(), wd, bd, final_conv_state=s1)
    b = mm.mamba_conv1d_fwd(xd[..., 101:103].contiguous(), wd, bd, conv_state=s1,
                            final_conv_state=s2)
    c = mm.mamba_conv1d_fwd(xd[..., 103:].contiguous(), wd, bd, conv_state=s2,
                            final_conv_state=s3)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([a, b, c], dim=-1), full)
    assert torch.equal(s3, xd[..., -3:])


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("width", [1, 4])
def test_conv_update_steps_equal_the_sequence(dtype, width):
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    x, w, bias, state = _inputs(dtype, 3, 96, 20, width, seed=7)
    xd, wd, bd, sd = to_dev(x, dtype), f32_dev(w), f32_dev(bias), to_dev(state, dtype)
    seq = mm.mamba_conv1d_fwd(xd, wd, bd, conv_state=sd if width > 1 else None)
    st = sd.clone()
    steps = [mm.mamba_conv1d_update(st, xd[..., t].contiguous(), wd, bd) for t in range(20)]
    torch.cuda.synchronize()
    assert torch.equal(torch.stack(steps, dim=-1), seq)
    if width > 1:
        assert torch.equal(st, xd[..., -(width - 1):])


def test_conv_full_size_sampled_rows():
    # the Mamba-2.8B layer shape (4 x 5120 channels x 2048 steps, width 4)
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    x, w, bias, _ = _inputs(synth.BF16, 4, 5120, 2048, 4, seed=9)
    out = mm.mamba_conv1d_fwd(to_dev(x, synth.BF16), f32_dev(w), f32_dev(bias))
    torch.cuda.synchronize()
    rows = synth.sample_rows(3, 4, 5120, 256)
    b, d = rows // 5120, rows % 5120
    xs = synth.widen(x, synth.BF16)[b, d][:, None, :]
    ref = np.concatenate([oracle.conv1d(xs[i:i + 1], w[d[i]:d[i] + 1], bias=bias[d[i]:d[i] + 1])[0]
                          for i in range(len(rows))], axis=0)[:, 0, :]
    got = to_f64(out.reshape(-1, 2048)[torch.from_numpy(rows).cuda()])
    assert_close(got, ref, synth.BF16, "conv out")


def test_conv_zero_length_copies_the_state():
    import selective_state_space_135_b300 as mm
    torch = torch_mod()
    x = torch.empty((2, 8, 0), dtype=torch.bfloat16, device="cuda")
    st = torch.randn((2, 8, 3), device="cuda").to(torch.bfloat16)
    fin = torch.zeros_like(st)
    mm.mamba_conv1d_fwd(x, torch.ones((8, 4), device="cuda"), None, conv_state=st,
                        final_conv_state=fin)
    torch.cuda.synchronize()
    assert torch.equal(fin, st)
