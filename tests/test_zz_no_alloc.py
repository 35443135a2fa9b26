"""GPU check of mamba_scan_fwd_noalloc, the scan entry point that allocates
nothing.  It is meant for callers that cannot allocate device memory (a
runtime that owns all of it in a fixed arena, or a latency-critical path
where an allocation may block or fail); its scratch is a fixed array inside
the library.

Two calls in a row, each compared bit for bit with mamba_scan_fwd on the
same inputs, through the C ABI: with the time chunks pinned, both entry
points run the same kernels on the same work units (the no-allocation one
only never uses the library's side stream, which changes where a pass runs,
not its arithmetic), so a wrong scratch offset or a stale read of the
shared array shows up as a difference in any bit.  The second call has a
different shape and a time-chunked plan, so stale contents of the shared
scratch from the first call would show up.  This file
sorts last so that a run that stops at the first failure has run every other
test before it.
"""

import pytest

import synth
from tests.gpu_util import f32_dev, to_dev, torch_mod

pytestmark = pytest.mark.gpu


def _inputs(shape):
    inp = synth.scan_inputs(shape)
    dt = shape.dtype
    return [to_dev(inp["u"], dt), to_dev(inp["delta"], dt), f32_dev(inp["dt_bias"]),
            f32_dev(inp["A"]), to_dev(inp["B"], dt), to_dev(inp["C"], dt),
            f32_dev(inp["D_skip"]), to_dev(inp["z"], dt)]


def _both(shape, chunks=0):
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    args = _inputs(shape)
    fin_shape = (shape.batch, shape.dim, shape.dstate)
    mm.mamba_scan_set_tuning(0, 0, chunks)
    try:
        fin_ref = torch.empty(fin_shape, device="cuda")
        y_ref = mm.mamba_scan_fwd(*args, True, final_state=fin_ref)
        fin = torch.full(fin_shape, float("nan"), device="cuda")
        y = torch.full_like(y_ref, float("nan"))
        mm.mamba_scan_fwd_noalloc(*args, True, y=y, final_state=fin)
        torch.cuda.synchronize()
    finally:
        mm.mamba_scan_set_tuning(0, 0, 0)
    return y, y_ref, fin, fin_ref


def test_noalloc_matches_scan_on_two_calls_in_a_row():
    import selective_state_space_135_b300 as mm
    first = synth.ScanShape("noalloc bf16 b2 d200 n16 l1024", 2, 200, 16, 1024, seed=91)
    second = synth.ScanShape("noalloc f32 b1 d70 n13 l600", 1, 70, 13, 600, dtype=synth.F32,
                             seed=92)
    torch = torch_mod()
    for shape, chunks in ((first, 0), (second, 3)):
        y, y_ref, fin, fin_ref = _both(shape, chunks)
        assert torch.equal(y, y_ref), "y differs from mamba_scan_fwd"
        assert torch.equal(fin, fin_ref), "final_state differs from mamba_scan_fwd"
    assert mm.mamba_device_status() == 0


def test_noalloc_rejects_a_problem_beyond_its_scratch():
    torch = torch_mod()
    import selective_state_space_135_b300 as mm
    # 1 x 140000 steps of packed B/C rows (128 bytes each) need 17.9 MB > 16 MiB
    L = 140000
    u = torch.zeros((1, 4, L), dtype=torch.bfloat16, device="cuda")
    Bm = torch.zeros((1, 16, L), dtype=torch.bfloat16, device="cuda")
    A = -torch.ones((4, 16), device="cuda")
    with pytest.raises(mm.MambaError) as err:
        mm.mamba_scan_fwd_noalloc(u, u.clone(), None, A, Bm, Bm.clone(), None, None, True,
                                  y=torch.empty_like(u))
    assert err.value.status == -9
