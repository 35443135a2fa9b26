"""The seeded input generators shared by the oracle and the kernels (CPU).

* bf16 rounding is round-to-nearest-even, checked bit for bit against
  torch's own float32 -> bfloat16 conversion, including ties, subnormals,
  infinities and NaN; widening is exact.
* The streams are deterministic per (seed, tensor name[, step]) and
  independent across names and steps.
* The workload recipe: shapes, dtypes, A = -(n + 1), dt_bias within its
  range, and the means and spreads of the normal draws.
* Row-wise streams (the million-step workload): any sampled rows equal the
  same rows of the full tensors.
"""

import numpy as np
import pytest

import synth


def test_bf16_round_matches_torch():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(0)
    x = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * 10.0,
        # exact ties between neighbouring bf16 values: 1 + k/128 + 1/256
        (1.0 + np.arange(64) / 128.0 + 1.0 / 256.0).astype(np.float32),
        np.array([0.0, -0.0, 1e-40, -1e-40, 3.0e38, np.inf, -np.inf], np.float32),
    ])
    ours = synth.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    nan = synth.bf16_round(np.array([np.nan], np.float32))
    assert np.isnan(synth.bf16_to_f32(nan))[0]


def test_widening_is_exact():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    wide = synth.bf16_to_f32(bits)
    finite = np.isfinite(wide)
    np.testing.assert_array_equal(synth.bf16_round(wide[finite]), bits[finite])
    np.testing.assert_array_equal(synth.widen(bits[finite], synth.BF16),
                                  wide[finite].astype(np.float64))


def test_streams_are_deterministic_and_independent():
    a = synth.normal(7, "u", (64, 64))
    b = synth.normal(7, "u", (64, 64))
    c = synth.normal(7, "delta", (64, 64))
    d = synth.normal(8, "u", (64, 64))
    e = synth.normal(7, "x", (64,), 1.0, 3)
    f = synth.normal(7, "x", (64,), 1.0, 4)
    np.testing.assert_array_equal(a, b)
    for other in (c, d):
        assert abs(np.corrcoef(a.ravel(), other.ravel())[0, 1]) < 0.05
    assert not np.array_equal(e, f)


def test_scan_recipe():
    shp = synth.ScanShape("t", 2, 64, 16, 512, dtype=synth.BF16, seed=3)
    inp = synth.scan_inputs(shp)
    for k in ("u", "delta", "z"):
        assert inp[k].shape == (2, 64, 512) and inp[k].dtype == np.uint16
    for k in ("B", "C"):
        assert inp[k].shape == (2, 16, 512) and inp[k].dtype == np.uint16
    np.testing.assert_array_equal(inp["A"], -np.tile(np.arange(1, 17, dtype=np.float32), (64, 1)))
    assert inp["dt_bias"].dtype == np.float32
    assert np.all((inp["dt_bias"] >= shp.dt_lo) & (inp["dt_bias"] <= shp.dt_hi))
    u = synth.widen(inp["u"], synth.BF16)
    dl = synth.widen(inp["delta"], synth.BF16)
    assert abs(u.mean()) < 0.02 and abs(u.std() - 1.0) < 0.02
    assert abs(dl.mean()) < 0.02 and abs(dl.std() - shp.delta_scale) < 0.02
    # the long workload's dt_bias range
    assert (synth.LONG.dt_lo, synth.LONG.dt_hi) == (-6.0, -4.0)
    again = synth.scan_inputs(shp)
    for k in ("u", "delta", "z", "B", "C", "dt_bias", "D_skip"):
        np.testing.assert_array_equal(inp[k], again[k])


def test_decode_steps_draw_fresh_inputs():
    shp = synth.DecodeShape("t", 4, 32, 16, 8)
    s0 = synth.decode_step_inputs(shp, 0)
    s1 = synth.decode_step_inputs(shp, 1)
    assert s0["x"].shape == (4, 32) and s0["B"].shape == (4, 16)
    assert not np.array_equal(s0["x"], s1["x"])
    np.testing.assert_array_equal(s0["x"], synth.decode_step_inputs(shp, 0)["x"])


def test_sample_rows():
    rows = synth.sample_rows(5, 4, 5120, 384)
    assert len(rows) == 384 and len(np.unique(rows)) == 384
    assert rows.min() >= 0 and rows.max() < 4 * 5120
    np.testing.assert_array_equal(rows, synth.sample_rows(5, 4, 5120, 384))
    assert len(synth.sample_rows(5, 1, 10, 50)) == 10


def test_rowwise_streams_sample_equals_full():
    # a row-wise shape draws every (batch, channel) row from its own stream:
    # a sampled sub-problem equals the same rows of the full tensors, rows do
    # not depend on the channel count, and the torch copy keeps the bits
    shp = synth.ScanShape("rowwise", 2, 9, 4, 40, rowwise=True, seed=17)
    full = synth.scan_inputs(shp)
    rows = np.array([9 + 2, 9 + 5, 9 + 8])       # batch entry 1, channels 2, 5, 8
    sub = synth.rowwise_sample(shp, rows)
    for k in ("u", "delta", "z"):
        assert np.array_equal(sub[k][0], full[k][1, [2, 5, 8]])
    assert np.array_equal(sub["B"][0], full["B"][1]) and np.array_equal(sub["C"][0], full["C"][1])
    assert np.array_equal(sub["A"], full["A"][[2, 5, 8]])
    assert np.array_equal(sub["dt_bias"], full["dt_bias"][[2, 5, 8]])
    wider = synth.ScanShape("rowwise", 2, 12, 4, 40, rowwise=True, seed=17)
    assert np.array_equal(synth.rows_block(wider, "u", 1, 2, 3)[0], full["u"][1, 2])
    again = synth.scan_inputs(shp)
    assert all(np.array_equal(again[k], full[k]) for k in ("u", "delta", "z", "B", "C"))
    import torch
    dev = synth.rowwise_to_device(shp, "delta", device="cpu", block_rows=4, threads=3)
    assert np.array_equal(dev.view(torch.int16).numpy().view(np.uint16), full["delta"])
    # the 0.5 scale of delta and unit scale of u
    assert abs(np.std(synth.widen(full["delta"], shp.dtype)) - 0.5) < 0.1
    assert abs(np.std(synth.widen(full["u"], shp.dtype)) - 1.0) < 0.2
