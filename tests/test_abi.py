"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/mamba_scan.h declares, and rejects bad arguments on
the host before touching the device."""

import os
import re

import numpy as np

import pytest

import selective_state_space_135_b300 as mm
from selective_state_space_135_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mamba_scan.h")

OK, ENULL, ESHAPE, EALIGN, ECUDA, ETIMEOUT, EALLOC, EDTYPE, EALIAS = 0, -1, -2, -3, -4, -5, -6, -7, -8
ETOOBIG = -9
EFLAGS = -10
EBOUNDS = -11
SOFTPLUS, ZOH, NOALLOC = 1, 2, 4


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mamba_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mamba_scan_fwd", "mamba_state_update", "mamba_status_string"):
        assert n in names
    assert set(names) == set(_lib.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_debug_library_exports_every_declared_symbol():
    # the build with index checks (MAMBA_SCAN_LIBRARY=debug) has the same ABI
    import ctypes
    path = os.path.join(os.path.dirname(_lib.lib_path()), "libmamba_scan_debug.so")
    assert os.path.exists(path), "build the library: python -m selective_state_space_135_b300.build"
    dbg = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(dbg, name), name


def test_status_strings(lib):
    for code in (OK, ENULL, ESHAPE, EALIGN, ECUDA, ETIMEOUT, EALLOC, EDTYPE, EALIAS, ETOOBIG,
                 EFLAGS, EBOUNDS):
        s = mm.mamba_status_string(code)
        assert s and s != "unknown status"
    assert mm.mamba_status_string(12345) == "unknown status"
    assert mm.mamba_version() >= 100


# Fake, well-aligned device addresses: validation must reject the call before
# anything dereferences them.
BASE = 1 << 40


def addr(i, extra=0):
    return BASE + i * (1 << 32) + extra


def scan_call(lib, batch=2, dim=16, dstate=4, seqlen=64, io=1, u=1, delta=2, dtb=3, A=4, B=5,
              C=6, Dk=7, z=8, softplus=1, y=9, fin=10, extra=None, fn="mamba_scan_fwd"):
    ptrs = dict(u=u, delta=delta, dtb=dtb, A=A, B=B, C=C, Dk=Dk, z=z, y=y, fin=fin)
    vals = {k: (None if v is None else addr(v, (extra or {}).get(k, 0))) for k, v in ptrs.items()}
    return getattr(lib, fn)(batch, dim, dstate, seqlen, io, vals["u"], vals["delta"],
                            vals["dtb"], vals["A"], vals["B"], vals["C"], vals["Dk"],
                            vals["z"], softplus, vals["y"], vals["fin"], None)


def test_scan_rejects_bad_shapes(lib):
    assert scan_call(lib, dstate=0) == ESHAPE
    assert scan_call(lib, dstate=17) == ESHAPE
    assert scan_call(lib, batch=0) == ESHAPE
    assert scan_call(lib, dim=0) == ESHAPE
    assert scan_call(lib, seqlen=-1) == ESHAPE
    assert scan_call(lib, io=5) == EDTYPE


def test_scan_rejects_null_required(lib):
    for k in ("u", "delta", "A", "B", "C", "y"):
        assert scan_call(lib, **{k: None}) == ENULL, k


def test_scan_rejects_misaligned(lib):
    # bf16 tensors need 2-byte alignment, fp32 ones 4-byte alignment
    assert scan_call(lib, extra={"u": 1}) == EALIGN
    assert scan_call(lib, extra={"y": 1}) == EALIGN
    assert scan_call(lib, io=0, extra={"B": 2}) == EALIGN
    assert scan_call(lib, extra={"A": 2}) == EALIGN
    assert scan_call(lib, extra={"fin": 2}) == EALIGN


def test_scan_rejects_aliasing(lib):
    assert scan_call(lib, y=1) == EALIAS        # y on top of u
    assert scan_call(lib, fin=4) == EALIAS      # final_state on top of A
    assert scan_call(lib, fin=9) == EALIAS      # final_state on top of y


def test_scan_nullable_inputs_pass_validation(lib):
    # With every nullable pointer absent the call passes validation.  seqlen 0
    # is a complete call that launches nothing (and writes nothing without a
    # final_state), so the fake addresses above are never dereferenced, on a
    # machine with or without a GPU.
    assert scan_call(lib, seqlen=0, dtb=None, Dk=None, z=None, fin=None) == OK


def test_noalloc_validates_like_the_scan(lib):
    fn = "mamba_scan_fwd_noalloc"
    assert scan_call(lib, dstate=17, fn=fn) == ESHAPE
    assert scan_call(lib, u=None, fn=fn) == ENULL
    assert scan_call(lib, extra={"u": 1}, fn=fn) == EALIGN
    assert scan_call(lib, y=1, fn=fn) == EALIAS


def test_noalloc_rejects_oversize_before_any_cuda_call(lib):
    # 2 x 70000 steps of packed B/C rows (128 bytes each at dstate 16) exceed
    # the 16 MiB fixed scratch; the check precedes every CUDA call
    fn = "mamba_scan_fwd_noalloc"
    assert scan_call(lib, dstate=16, seqlen=70000, fn=fn) == ETOOBIG
    assert scan_call(lib, dstate=4, seqlen=300000, fn=fn) == ETOOBIG
    assert "MAMBA_NOALLOC_SCRATCH_BYTES" in mm.mamba_status_string(ETOOBIG)


def ex_call(lib, batch=2, dim=16, dstate=4, seqlen=64, io=1, flags=SOFTPLUS, h0=11, lens=12,
            fin=10, y=9, extra=None):
    ptrs = dict(u=1, delta=2, dtb=3, A=4, B=5, C=6, Dk=7, z=8, y=y, fin=fin, h0=h0, lens=lens)
    v = {k: (None if q is None else addr(q, (extra or {}).get(k, 0))) for k, q in ptrs.items()}
    return lib.mamba_scan_fwd_ex(batch, dim, dstate, seqlen, io, v["u"], v["delta"], v["dtb"],
                                 v["A"], v["B"], v["C"], v["Dk"], v["z"], flags, v["h0"],
                                 v["lens"], v["y"], v["fin"], None)


def test_scan_ex_validation(lib):
    assert ex_call(lib, flags=8) == EFLAGS
    assert ex_call(lib, flags=-1) == EFLAGS
    assert ex_call(lib, dstate=17) == ESHAPE
    assert ex_call(lib, extra={"h0": 2}) == EALIGN
    assert ex_call(lib, extra={"lens": 2}) == EALIGN
    assert ex_call(lib, h0=9) == EALIAS           # initial state on top of y
    assert ex_call(lib, h0=10) == EALIAS          # initial state on top of final_state
    assert ex_call(lib, lens=9) == EALIAS         # lengths on top of y
    assert ex_call(lib, flags=NOALLOC, dstate=16, seqlen=70000) == ETOOBIG


def test_scan_ex_passes_validation_without_launching(lib):
    # seqlen 0 with no final_state is complete without any CUDA call, so the
    # fake addresses are never dereferenced
    for flags in (0, SOFTPLUS, ZOH, SOFTPLUS | ZOH | NOALLOC):
        assert ex_call(lib, seqlen=0, flags=flags, fin=None) == OK


def step_call(lib, batch=2, dim=8, dstate=16, io=1, state=1, x=2, delta=3, dtb=4, A=5, B=6, C=7,
              Dk=8, z=9, y=10, extra=None):
    ptrs = dict(state=state, x=x, delta=delta, dtb=dtb, A=A, B=B, C=C, Dk=Dk, z=z, y=y)
    vals = {k: (None if v is None else addr(v, (extra or {}).get(k, 0))) for k, v in ptrs.items()}
    return lib.mamba_state_update(batch, dim, dstate, io, vals["state"], vals["x"], vals["delta"],
                                  vals["dtb"], vals["A"], vals["B"], vals["C"], vals["Dk"],
                                  vals["z"], vals["y"], None)


def test_state_update_validation(lib):
    assert step_call(lib, dstate=17) == ESHAPE
    assert step_call(lib, batch=0) == ESHAPE
    assert step_call(lib, io=2) == EDTYPE
    for k in ("state", "x", "delta", "A", "B", "C", "y"):
        assert step_call(lib, **{k: None}) == ENULL, k
    assert step_call(lib, extra={"state": 2}) == EALIGN
    assert step_call(lib, extra={"x": 1}) == EALIGN
    assert step_call(lib, y=1) == EALIAS
    assert step_call(lib, x=1) == EALIAS       # state overlaps x


def bwd_call(lib, flags=SOFTPLUS, dstate=16, extra=None, **over):
    names = ("u", "delta", "dtb", "A", "B", "C", "Dk", "z", "h0", "dy", "dfin", "du", "ddelta",
             "dA", "dB", "dC", "dD", "dz", "dbias", "dh0")
    v = {k: addr(i, (extra or {}).get(k, 0)) for i, k in enumerate(names, 1)}
    v.update(over)
    return lib.mamba_scan_bwd(2, 16, dstate, 64, 1, v["u"], v["delta"], v["dtb"], v["A"], v["B"],
                              v["C"], v["Dk"], v["z"], flags, v["h0"], v["dy"], v["dfin"],
                              v["du"], v["ddelta"], v["dA"], v["dB"], v["dC"], v["dD"], v["dz"],
                              v["dbias"], v["dh0"], None)


def test_scan_bwd_validation(lib):
    # every case is rejected on the host, before any CUDA call
    assert bwd_call(lib, flags=ZOH) == EFLAGS
    assert bwd_call(lib, flags=SOFTPLUS | NOALLOC) == EFLAGS
    assert bwd_call(lib, dstate=17) == ESHAPE
    for k in ("u", "delta", "A", "B", "C", "dy", "du", "ddelta", "dA", "dB", "dC"):
        assert bwd_call(lib, **{k: None}) == ENULL, k
    assert bwd_call(lib, dz=None) == ENULL            # z given without dz
    assert bwd_call(lib, extra={"du": 1}) == EALIGN
    assert bwd_call(lib, extra={"dA": 2}) == EALIGN
    assert bwd_call(lib, du=addr(1)) == EALIAS        # du on top of u
    assert bwd_call(lib, dB=addr(14)) == EALIAS       # dB on top of dA
    assert bwd_call(lib, dh0=addr(9)) == EALIAS       # d_initial_state on top of initial_state


def test_conv1d_validation(lib):
    # rejected on the host, before any CUDA call
    def fwd(width=4, **kw):
        v = dict(x=addr(1), w=addr(2), b=addr(3), st=addr(4), out=addr(5), fin=addr(6))
        v.update(kw)
        return lib.mamba_conv1d_fwd(2, 16, 64, width, 1, v["x"], v["w"], v["b"], v["st"], 1,
                                    v["out"], v["fin"], None)
    assert fwd(width=0) == ESHAPE
    assert fwd(width=9) == ESHAPE
    assert fwd(x=None) == ENULL
    assert fwd(w=None) == ENULL
    assert fwd(out=addr(1)) == EALIAS            # out on top of x
    assert fwd(fin=addr(4)) == EALIAS            # final state on top of the state
    assert fwd(w=addr(2) + 2) == EALIGN
    assert fwd(x=addr(1) + 1) == EALIGN

    def upd(width=4, **kw):
        v = dict(st=addr(1), x=addr(2), w=addr(3), b=addr(4), out=addr(5))
        v.update(kw)
        return lib.mamba_conv1d_update(2, 16, width, 1, v["st"], v["x"], v["w"], v["b"], 1,
                                       v["out"], None)
    assert upd(width=9) == ESHAPE
    assert upd(st=None) == ENULL
    assert upd(out=addr(2)) == EALIAS


def test_state_update_ex_flags(lib):
    def call(flags, **kw):
        v = {k: addr(i) for i, k in enumerate(("state", "x", "delta", "dtb", "A", "B", "C",
                                               "Dk", "z", "y"), 1)}
        v.update(kw)
        return lib.mamba_state_update_ex(2, 8, 16, 1, v["state"], v["x"], v["delta"], v["dtb"],
                                         v["A"], v["B"], v["C"], v["Dk"], v["z"], flags, v["y"],
                                         None)
    assert call(NOALLOC) == EFLAGS
    assert call(16) == EFLAGS
    assert call(SOFTPLUS | ZOH, state=None) == ENULL
    assert call(ZOH, y=addr(1)) == EALIAS


def test_tuning_validation(lib):
    assert lib.mamba_scan_set_tuning(4, 0, 0, 0) == ESHAPE
    assert lib.mamba_scan_set_tuning(-1, 0, 0, 0) == ESHAPE
    assert lib.mamba_scan_set_tuning(3, 0, 0, 0) == OK
    assert lib.mamba_scan_set_tuning(0, 9, 0, 0) == ESHAPE
    assert lib.mamba_scan_set_tuning(0, 0, -1, 0) == ESHAPE
    assert lib.mamba_scan_set_tuning(0, 0, 0, 3) == ESHAPE
    assert lib.mamba_scan_set_tuning(0, 0, 0, -1) == ESHAPE
    assert lib.mamba_scan_set_tuning(0, 0, 0, 2) == OK
    assert lib.mamba_scan_set_tuning(0, 0, 0, 0) == OK


def test_selftest_rejects_bad_limits(lib):
    # checked before anything is launched
    assert lib.mamba_selftest_wait_timeout(0, None) == ESHAPE
    assert lib.mamba_selftest_wait_timeout(3000000, None) == ESHAPE


def test_profiler_without_launches(lib):
    mm.mamba_profile_begin()
    prof = mm.mamba_profile_end()
    assert set(prof) == set(_lib.KIND_NAMES)
    assert all(v == (0.0, 0) for v in prof.values())


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    u = torch.zeros(1, 4, 8)
    with pytest.raises(ValueError):
        mm.mamba_scan_fwd(u, u, None, torch.zeros(4, 2), torch.zeros(1, 2, 8),
                          torch.zeros(1, 2, 8), None, None)


def test_header_is_plain_c(tmp_path):
    # The boundary is a C ABI: a C11 translation unit that includes the
    # header and takes the address of every entry point must compile and link
    # against the library, with no C++ or torch types involved.
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if gcc is None or not os.path.isdir(cuda_inc):
        pytest.skip("gcc or the CUDA headers are not available")
    names = declared_functions()
    src = tmp_path / "abi_check.c"
    src.write_text('#include "mamba_scan.h"\n#include <stdio.h>\n'
                   "int main(void) {\n    const void* fns[] = {\n"
                   + "".join(f"        (const void*)&{n},\n" for n in names)
                   + "    };\n    printf(\"%d\\n\", (int)(sizeof(fns) / sizeof(fns[0])));\n"
                   "    return 0;\n}\n")
    exe = tmp_path / "abi_check"
    lib = _lib.lib_path()
    cmd = [gcc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
           str(src), "-o", str(exe), lib, f"-Wl,-rpath,{os.path.dirname(lib)}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_checkpoint_bytes(lib):
    # batch * dim * ceil(seqlen / 12) * padded dstate * 4 bytes
    assert lib.mamba_scan_checkpoint_bytes(2, 16, 4, 64) == 2 * 16 * 6 * 4 * 4
    assert lib.mamba_scan_checkpoint_bytes(1, 3, 5, 12) == 1 * 3 * 1 * 8 * 4
    assert lib.mamba_scan_checkpoint_bytes(1, 3, 16, 13) == 1 * 3 * 2 * 16 * 4
    assert lib.mamba_scan_checkpoint_bytes(1, 3, 16, 0) == 0
    assert lib.mamba_scan_checkpoint_bytes(1, 3, 17, 10) == -1
    assert lib.mamba_scan_checkpoint_bytes(0, 3, 4, 10) == -1
    for b, d, n, l in ((2, 16, 4, 64), (1, 3, 5, 12), (3, 7, 16, 25)):
        shp = _lib.checkpoint_shape(b, d, n, l)
        assert lib.mamba_scan_checkpoint_bytes(b, d, n, l) == 4 * int(np.prod(shp))


def train_call(lib, flags=SOFTPLUS, extra=None, **over):
    names = ("u", "delta", "dtb", "A", "B", "C", "Dk", "z", "h0", "y", "fin", "ckpt")
    v = {k: addr(i, (extra or {}).get(k, 0)) for i, k in enumerate(names, 1)}
    v.update(over)
    return lib.mamba_scan_fwd_train(2, 16, 16, 64, 1, v["u"], v["delta"], v["dtb"], v["A"],
                                    v["B"], v["C"], v["Dk"], v["z"], flags, v["h0"], v["y"],
                                    v["fin"], v["ckpt"], None)


def test_scan_fwd_train_validation(lib):
    # every case is rejected on the host, before any CUDA call
    assert train_call(lib, flags=ZOH) == EFLAGS
    assert train_call(lib, flags=SOFTPLUS | NOALLOC) == EFLAGS
    for k in ("u", "delta", "A", "B", "C", "y", "ckpt"):
        assert train_call(lib, **{k: None}) == ENULL, k
    assert train_call(lib, extra={"ckpt": 8}) == EALIGN     # checkpoints need 16 bytes
    assert train_call(lib, ckpt=addr(1)) == EALIAS          # on top of u
    assert train_call(lib, ckpt=addr(10)) == EALIAS         # on top of y
    assert train_call(lib, ckpt=addr(11)) == EALIAS         # on top of final_state


def test_scan_bwd_ckpt_validation(lib):
    def call(**over):
        names = ("u", "delta", "dtb", "A", "B", "C", "Dk", "z", "ckpt", "dy", "dfin", "du",
                 "ddelta", "dA", "dB", "dC", "dD", "dz", "dbias", "dh0")
        flags = over.pop("flags", SOFTPLUS)
        extra = over.pop("extra", {})
        v = {k: addr(i, extra.get(k, 0)) for i, k in enumerate(names, 1)}
        v.update(over)
        return lib.mamba_scan_bwd_ckpt(2, 16, 16, 64, 1, *(v[k] for k in names[:8]), flags,
                                       *(v[k] for k in names[8:]), None)
    assert call(flags=ZOH) == EFLAGS
    assert call(ckpt=None) == ENULL
    for k in ("u", "dy", "du", "dB"):
        assert call(**{k: None}) == ENULL, k
    assert call(extra={"ckpt": 4}) == EALIGN
    assert call(du=addr(9)) == EALIAS                 # du on top of the checkpoints
    assert call(dh0=addr(9)) == EALIAS                # d_initial_state on top of them
