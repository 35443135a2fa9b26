"""ctypes marshalling for libmamba_scan.so (see include/mamba_scan.h)."""

from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
# MAMBA_SCAN_LIBRARY=debug selects the build whose kernels check the index
# of every global access (same entry points, same results)
_LIB = os.path.join(HERE, "libmamba_scan_debug.so" if os.environ.get("MAMBA_SCAN_LIBRARY") == "debug"
                    else "libmamba_scan.so")
_lock = threading.Lock()
_lib = None

MAMBA_F32 = 0
MAMBA_BF16 = 1

# every symbol the header declares
EXPORTS = ("mamba_scan_fwd", "mamba_scan_fwd_noalloc", "mamba_scan_fwd_ex", "mamba_scan_bwd",
           "mamba_conv1d_fwd", "mamba_conv1d_update", "mamba_state_update",
           "mamba_state_update_ex", "mamba_status_string", "mamba_device_status",
           "mamba_selftest_wait_timeout", "mamba_version", "mamba_scan_set_tuning",
           "mamba_profile_begin", "mamba_profile_end", "mamba_probe_pipe_rate",
           "mamba_debug_build", "mamba_selftest_bounds", "mamba_scan_checkpoint_bytes",
           "mamba_scan_fwd_train", "mamba_scan_bwd_ckpt")

# flags of the extended entry points
MAMBA_FLAG_SOFTPLUS = 1
MAMBA_FLAG_ZOH = 2
MAMBA_FLAG_NOALLOC = 4

KIND_NAMES = ("scan", "chunk_summary", "chunk_carry", "state_update", "pack_bc",
              "bwd_checkpoint", "bwd", "bwd_reduce", "conv1d", "bwd_summary")


class MambaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {mamba_status_string(status)} (status {status})")


def lib_path() -> str:
    return _LIB


def load():
    """Load the CUDA library; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB):
            raise ImportError(
                f"{_LIB} is missing: build it with `python -m selective_state_space_135_b300.build`")
        lib = ctypes.CDLL(_LIB)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.mamba_scan_fwd.argtypes = [i64, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                       i32, vp, vp, vp]
        lib.mamba_scan_fwd.restype = i32
        lib.mamba_scan_fwd_noalloc.argtypes = lib.mamba_scan_fwd.argtypes
        lib.mamba_scan_fwd_noalloc.restype = i32
        lib.mamba_state_update.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                           vp, vp, vp]
        lib.mamba_state_update.restype = i32
        lib.mamba_scan_fwd_ex.argtypes = [i64, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                          i32, vp, vp, vp, vp, vp]
        lib.mamba_scan_fwd_ex.restype = i32
        lib.mamba_state_update_ex.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                              vp, i32, vp, vp]
        lib.mamba_state_update_ex.restype = i32
        # sizes, dtype; 8 inputs; flags; initial state, dy, d_final_state;
        # 9 outputs; stream
        lib.mamba_scan_bwd.argtypes = [i64, i64, i64, i64, i32] + [vp] * 8 + [i32] + [vp] * 3 \
            + [vp] * 9 + [vp]
        lib.mamba_scan_bwd.restype = i32
        lib.mamba_scan_bwd_ckpt.argtypes = lib.mamba_scan_bwd.argtypes   # checkpoints for h0
        lib.mamba_scan_bwd_ckpt.restype = i32
        lib.mamba_scan_checkpoint_bytes.argtypes = [i64, i64, i64, i64]
        lib.mamba_scan_checkpoint_bytes.restype = i64
        lib.mamba_scan_fwd_train.argtypes = [i64, i64, i64, i64, i32] + [vp] * 8 + [i32] \
            + [vp] * 4 + [vp]
        lib.mamba_scan_fwd_train.restype = i32
        lib.mamba_conv1d_fwd.argtypes = [i64, i64, i64, i32, i32, vp, vp, vp, vp, i32, vp, vp, vp]
        lib.mamba_conv1d_fwd.restype = i32
        lib.mamba_conv1d_update.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, i32, vp, vp]
        lib.mamba_conv1d_update.restype = i32
        lib.mamba_status_string.argtypes = [i32]
        lib.mamba_status_string.restype = ctypes.c_char_p
        lib.mamba_device_status.argtypes = [vp]
        lib.mamba_device_status.restype = i32
        lib.mamba_selftest_wait_timeout.argtypes = [i64, vp]
        lib.mamba_selftest_wait_timeout.restype = i32
        lib.mamba_version.argtypes = []
        lib.mamba_version.restype = i32
        lib.mamba_scan_set_tuning.argtypes = [i32, i32, i32, i32]
        lib.mamba_scan_set_tuning.restype = i32
        lib.mamba_profile_begin.argtypes = []
        lib.mamba_profile_begin.restype = i32
        lib.mamba_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_int64), i32]
        lib.mamba_profile_end.restype = i32
        lib.mamba_probe_pipe_rate.argtypes = [i32, i32, i32, i64,
                                              ctypes.POINTER(ctypes.c_double),
                                              ctypes.POINTER(ctypes.c_double), vp]
        lib.mamba_probe_pipe_rate.restype = i32
        lib.mamba_debug_build.argtypes = [ctypes.POINTER(ctypes.c_int)]
        lib.mamba_debug_build.restype = i32
        lib.mamba_selftest_bounds.argtypes = [vp]
        lib.mamba_selftest_bounds.restype = i32
        _lib = lib
        return lib


def mamba_status_string(status: int) -> str:
    return load().mamba_status_string(int(status)).decode()


def mamba_version() -> int:
    return load().mamba_version()


def _torch():
    import torch
    return torch


def _io_dtype(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return MAMBA_F32
    if t.dtype == torch.bfloat16:
        return MAMBA_BF16
    raise TypeError(f"unsupported io dtype {t.dtype}; use float32 or bfloat16")


def _ptr(t, name, dtype=None, shape=None, device=None):
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr() or None


def _stream_handle(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _scan_call(fn_name, u, delta, dt_bias, A, B, C, D_skip, z, softplus, y, final_state,
               stream):
    torch = _torch()
    lib = load()
    batch, dim, L = u.shape
    N = A.shape[1]
    dev = u.device
    io = _io_dtype(u)
    if y is None:
        y = torch.empty_like(u)
    args = (
        _ptr(u, "u", u.dtype, (batch, dim, L), dev),
        _ptr(delta, "delta", u.dtype, (batch, dim, L), dev),
        _ptr(dt_bias, "dt_bias", torch.float32, (dim,), dev),
        _ptr(A, "A", torch.float32, (dim, N), dev),
        _ptr(B, "B", u.dtype, (batch, N, L), dev),
        _ptr(C, "C", u.dtype, (batch, N, L), dev),
        _ptr(D_skip, "D_skip", torch.float32, (dim,), dev),
        _ptr(z, "z", u.dtype, (batch, dim, L), dev),
    )
    yp = _ptr(y, "y", u.dtype, (batch, dim, L), dev)
    fp = _ptr(final_state, "final_state", torch.float32, (batch, dim, N), dev)
    with torch.cuda.device(dev):
        st = _stream_handle(stream, dev)
        rc = getattr(lib, fn_name)(batch, dim, N, L, io, args[0], args[1], args[2], args[3],
                                   args[4], args[5], args[6], args[7], int(bool(softplus)),
                                   yp, fp, st)
    if rc != 0:
        raise MambaError(rc, fn_name)
    return y


def mamba_scan_fwd(u, delta, dt_bias, A, B, C, D_skip, z, softplus: bool = True,
                   y=None, final_state=None, stream=None):
    """Selective scan.  u, delta, z: (batch, dim, L); B, C: (batch, N, L);
    A: (dim, N) fp32; dt_bias, D_skip: (dim,) fp32 or None; z may be None.
    y (allocated if None) gets the output; final_state (batch, dim, N) fp32,
    if given, gets the state after the last step.  Returns y.
    """
    return _scan_call("mamba_scan_fwd", u, delta, dt_bias, A, B, C, D_skip, z, softplus, y,
                      final_state, stream)


def mamba_scan_fwd_noalloc(u, delta, dt_bias, A, B, C, D_skip, z, softplus: bool = True,
                           y=None, final_state=None, stream=None):
    """mamba_scan_fwd through the entry point that allocates no scratch: the
    library uses its fixed device array (MAMBA_NOALLOC_SCRATCH_BYTES) instead.
    Same arguments; pass y to keep the call free of allocations here as well.
    Calls that overlap on the GPU share that array and must be serialised."""
    return _scan_call("mamba_scan_fwd_noalloc", u, delta, dt_bias, A, B, C, D_skip, z, softplus,
                      y, final_state, stream)


def scan_flags(softplus: bool = True, zoh: bool = False, no_alloc: bool = False) -> int:
    return ((MAMBA_FLAG_SOFTPLUS if softplus else 0) | (MAMBA_FLAG_ZOH if zoh else 0)
            | (MAMBA_FLAG_NOALLOC if no_alloc else 0))


def mamba_scan_fwd_ex(u, delta, dt_bias, A, B, C, D_skip, z, softplus: bool = True,
                      zoh: bool = False, initial_state=None, seqlens=None, y=None,
                      final_state=None, no_alloc: bool = False, stream=None):
    """mamba_scan_fwd plus an initial state (batch, dim, N) fp32, per-entry
    lengths seqlens (batch,) int32 on the device, the zero-order-hold input
    term (zoh=True) and the no-allocation scratch (no_alloc=True).  Returns y;
    y[b, :, t] is 0 for t >= seqlens[b]."""
    torch = _torch()
    lib = load()
    batch, dim, L = u.shape
    N = A.shape[1]
    dev = u.device
    io = _io_dtype(u)
    if y is None:
        y = torch.empty_like(u)
    args = (
        _ptr(u, "u", u.dtype, (batch, dim, L), dev),
        _ptr(delta, "delta", u.dtype, (batch, dim, L), dev),
        _ptr(dt_bias, "dt_bias", torch.float32, (dim,), dev),
        _ptr(A, "A", torch.float32, (dim, N), dev),
        _ptr(B, "B", u.dtype, (batch, N, L), dev),
        _ptr(C, "C", u.dtype, (batch, N, L), dev),
        _ptr(D_skip, "D_skip", torch.float32, (dim,), dev),
        _ptr(z, "z", u.dtype, (batch, dim, L), dev),
    )
    hp = _ptr(initial_state, "initial_state", torch.float32, (batch, dim, N), dev)
    lp = _ptr(seqlens, "seqlens", torch.int32, (batch,), dev)
    yp = _ptr(y, "y", u.dtype, (batch, dim, L), dev)
    fp = _ptr(final_state, "final_state", torch.float32, (batch, dim, N), dev)
    with torch.cuda.device(dev):
        st = _stream_handle(stream, dev)
        rc = lib.mamba_scan_fwd_ex(batch, dim, N, L, io, args[0], args[1], args[2], args[3],
                                   args[4], args[5], args[6], args[7],
                                   scan_flags(softplus, zoh, no_alloc), hp, lp, yp, fp, st)
    if rc != 0:
        raise MambaError(rc, "mamba_scan_fwd_ex")
    return y


def mamba_scan_bwd(u, delta, dt_bias, A, B, C, D_skip, z, dy, softplus: bool = True,
                   initial_state=None, d_final_state=None, want_initial_state_grad: bool = False,
                   out=None, stream=None) -> dict:
    """Backward pass of the scan: returns a dict of gradients du, ddelta, dz
    (None without z), dA, dB, dC, dD_skip, ddt_bias and, when asked,
    d_initial_state.  dy has u's shape and dtype; d_final_state (batch, dim,
    N) fp32 is optional.  `out` may supply any of the output tensors."""
    batch, dim, _ = u.shape
    h0 = _ptr(initial_state, "initial_state", _torch().float32, (batch, dim, A.shape[1]),
              u.device)
    return _bwd_call("mamba_scan_bwd", h0, u, delta, dt_bias, A, B, C, D_skip, z, dy, softplus,
                     d_final_state, want_initial_state_grad, out, stream)


def mamba_scan_checkpoint_bytes(batch: int, dim: int, dstate: int, seqlen: int) -> int:
    """Bytes of the state checkpoints of mamba_scan_fwd_train (-1: bad shape)."""
    return int(load().mamba_scan_checkpoint_bytes(batch, dim, dstate, seqlen))


def checkpoint_shape(batch: int, dim: int, dstate: int, seqlen: int) -> tuple:
    """(batch, ceil(seqlen / 12), P / 4, dim, 4) fp32 with P = dstate padded to
    4, 8 or 16: entries in quads of four, channel-major within a quad."""
    pad = 4 if dstate <= 4 else (8 if dstate <= 8 else 16)
    return (batch, (seqlen + 11) // 12, pad // 4, dim, 4)


def mamba_scan_fwd_train(u, delta, dt_bias, A, B, C, D_skip, z, softplus: bool = True,
                         initial_state=None, y=None, final_state=None, checkpoints=None,
                         stream=None):
    """The forward of a training step: y (and final_state) as mamba_scan_fwd_ex
    from initial_state, plus the state checkpoints that mamba_scan_bwd_ckpt
    reads (allocated if None, shape checkpoint_shape(...)).  Returns
    (y, checkpoints)."""
    torch = _torch()
    lib = load()
    batch, dim, L = u.shape
    N = A.shape[1]
    dev = u.device
    io = _io_dtype(u)
    if y is None:
        y = torch.empty_like(u)
    cks = checkpoint_shape(batch, dim, N, L)
    if checkpoints is None:
        checkpoints = torch.empty(cks, dtype=torch.float32, device=dev)
    args = (
        _ptr(u, "u", u.dtype, (batch, dim, L), dev),
        _ptr(delta, "delta", u.dtype, (batch, dim, L), dev),
        _ptr(dt_bias, "dt_bias", torch.float32, (dim,), dev),
        _ptr(A, "A", torch.float32, (dim, N), dev),
        _ptr(B, "B", u.dtype, (batch, N, L), dev),
        _ptr(C, "C", u.dtype, (batch, N, L), dev),
        _ptr(D_skip, "D_skip", torch.float32, (dim,), dev),
        _ptr(z, "z", u.dtype, (batch, dim, L), dev),
    )
    hp = _ptr(initial_state, "initial_state", torch.float32, (batch, dim, N), dev)
    yp = _ptr(y, "y", u.dtype, (batch, dim, L), dev)
    fp = _ptr(final_state, "final_state", torch.float32, (batch, dim, N), dev)
    cp = _ptr(checkpoints, "checkpoints", torch.float32, cks, dev)
    with torch.cuda.device(dev):
        st = _stream_handle(stream, dev)
        rc = lib.mamba_scan_fwd_train(batch, dim, N, L, io, *args,
                                      scan_flags(softplus), hp, yp, fp, cp, st)
    if rc != 0:
        raise MambaError(rc, "mamba_scan_fwd_train")
    return y, checkpoints


def mamba_scan_bwd_ckpt(u, delta, dt_bias, A, B, C, D_skip, z, dy, checkpoints,
                        softplus: bool = True, d_final_state=None,
                        want_initial_state_grad: bool = False, out=None, stream=None) -> dict:
    """mamba_scan_bwd from the checkpoints of mamba_scan_fwd_train on the same
    inputs (the initial state is inside them).  Same results, bit for bit."""
    batch, dim, L = u.shape
    cp = _ptr(checkpoints, "checkpoints", _torch().float32,
              checkpoint_shape(batch, dim, A.shape[1], L), u.device)
    return _bwd_call("mamba_scan_bwd_ckpt", cp, u, delta, dt_bias, A, B, C, D_skip, z, dy,
                     softplus, d_final_state, want_initial_state_grad, out, stream)


def _bwd_call(fn_name, state_ptr, u, delta, dt_bias, A, B, C, D_skip, z, dy, softplus,
              d_final_state, want_initial_state_grad, out, stream) -> dict:
    torch = _torch()
    lib = load()
    batch, dim, L = u.shape
    N = A.shape[1]
    dev = u.device
    io = _io_dtype(u)
    f32 = torch.float32
    o = dict(out or {})
    o.setdefault("du", torch.empty_like(u))
    o.setdefault("ddelta", torch.empty_like(u))
    o.setdefault("dz", None if z is None else torch.empty_like(u))
    o.setdefault("dA", torch.empty((dim, N), dtype=f32, device=dev))
    o.setdefault("dB", torch.empty((batch, N, L), dtype=f32, device=dev))
    o.setdefault("dC", torch.empty((batch, N, L), dtype=f32, device=dev))
    o.setdefault("dD_skip", torch.empty((dim,), dtype=f32, device=dev))
    o.setdefault("ddt_bias", torch.empty((dim,), dtype=f32, device=dev))
    o.setdefault("d_initial_state", torch.empty((batch, dim, N), dtype=f32, device=dev)
                 if want_initial_state_grad else None)
    ins = (
        _ptr(u, "u", u.dtype, (batch, dim, L), dev),
        _ptr(delta, "delta", u.dtype, (batch, dim, L), dev),
        _ptr(dt_bias, "dt_bias", f32, (dim,), dev),
        _ptr(A, "A", f32, (dim, N), dev),
        _ptr(B, "B", u.dtype, (batch, N, L), dev),
        _ptr(C, "C", u.dtype, (batch, N, L), dev),
        _ptr(D_skip, "D_skip", f32, (dim,), dev),
        _ptr(z, "z", u.dtype, (batch, dim, L), dev),
    )
    dyp = _ptr(dy, "dy", u.dtype, (batch, dim, L), dev)
    dfp = _ptr(d_final_state, "d_final_state", f32, (batch, dim, N), dev)
    shapes = dict(du=((batch, dim, L), u.dtype), ddelta=((batch, dim, L), u.dtype),
                  dz=((batch, dim, L), u.dtype), dA=((dim, N), f32), dB=((batch, N, L), f32),
                  dC=((batch, N, L), f32), dD_skip=((dim,), f32), ddt_bias=((dim,), f32),
                  d_initial_state=((batch, dim, N), f32))
    op = {k: _ptr(o[k], k, shapes[k][1], shapes[k][0], dev) for k in shapes}
    with torch.cuda.device(dev):
        st = _stream_handle(stream, dev)
        rc = getattr(lib, fn_name)(batch, dim, N, L, io, *ins, int(bool(softplus)), state_ptr,
                                   dyp, dfp, op["du"], op["ddelta"], op["dA"], op["dB"],
                                   op["dC"], op["dD_skip"], op["dz"], op["ddt_bias"],
                                   op["d_initial_state"], st)
    if rc != 0:
        raise MambaError(rc, fn_name)
    return o


def mamba_conv1d_fwd(x, weight, bias=None, conv_state=None, silu: bool = True, out=None,
                     final_conv_state=None, stream=None):
    """Causal depthwise convolution (+ SiLU).  x: (batch, dim, L); weight:
    (dim, W) fp32; bias (dim,) fp32 or None; conv_state (batch, dim, W-1) in
    x's dtype or None; final_conv_state, if given, gets the W-1 last inputs.
    Returns out (allocated if None)."""
    torch = _torch()
    lib = load()
    batch, dim, L = x.shape
    W = weight.shape[1]
    dev = x.device
    io = _io_dtype(x)
    if out is None:
        out = torch.empty_like(x)
    args = (_ptr(x, "x", x.dtype, (batch, dim, L), dev),
            _ptr(weight, "weight", torch.float32, (dim, W), dev),
            _ptr(bias, "bias", torch.float32, (dim,), dev),
            _ptr(conv_state, "conv_state", x.dtype, (batch, dim, W - 1), dev))
    op = _ptr(out, "out", x.dtype, (batch, dim, L), dev)
    fp = _ptr(final_conv_state, "final_conv_state", x.dtype, (batch, dim, W - 1), dev)
    with torch.cuda.device(dev):
        st = _stream_handle(stream, dev)
        rc = lib.mamba_conv1d_fwd(batch, dim, L, W, io, *args, int(bool(silu)), op, fp, st)
    if rc != 0:
        raise MambaError(rc, "mamba_conv1d_fwd")
    return out


def mamba_conv1d_update(conv_state, x, weight, bias=None, silu: bool = True, out=None,
                        stream=None):
    """One generation step of the convolution; conv_state (batch, dim, W-1)
    is updated in place.  x: (batch, dim).  Returns out (batch, dim)."""
    torch = _torch()
    lib = load()
    batch, dim = x.shape
    W = weight.shape[1]
    dev = x.device
    io = _io_dtype(x)
    if out is None:
        out = torch.empty_like(x)
    sp = _ptr(conv_state, "conv_state", x.dtype, (batch, dim, W - 1), dev) if W > 1 else None
    args = (_ptr(x, "x", x.dtype, (batch, dim), dev),
            _ptr(weight, "weight", torch.float32, (dim, W), dev),
            _ptr(bias, "bias", torch.float32, (dim,), dev))
    op = _ptr(out, "out", x.dtype, (batch, dim), dev)
    with torch.cuda.device(dev):
        st = _stream_handle(stream, dev)
        rc = lib.mamba_conv1d_update(batch, dim, W, io, sp, *args, int(bool(silu)), op, st)
    if rc != 0:
        raise MambaError(rc, "mamba_conv1d_update")
    return out


def mamba_state_update(state, x, delta, dt_bias, A, B, C, D_skip, z, y=None, stream=None):
    """One decode step in place on state (batch, dim, N) fp32.  x, delta, z:
    (batch, dim); B, C: (batch, N).  Returns y (batch, dim)."""
    torch = _torch()
    lib = load()
    batch, dim, N = state.shape
    dev = state.device
    io = _io_dtype(x)
    if y is None:
        y = torch.empty_like(x)
    sp = _ptr(state, "state", torch.float32, (batch, dim, N), dev)
    args = (
        _ptr(x, "x", x.dtype, (batch, dim), dev),
        _ptr(delta, "delta", x.dtype, (batch, dim), dev),
        _ptr(dt_bias, "dt_bias", torch.float32, (dim,), dev),
        _ptr(A, "A", torch.float32, (dim, N), dev),
        _ptr(B, "B", x.dtype, (batch, N), dev),
        _ptr(C, "C", x.dtype, (batch, N), dev),
        _ptr(D_skip, "D_skip", torch.float32, (dim,), dev),
        _ptr(z, "z", x.dtype, (batch, dim), dev),
    )
    yp = _ptr(y, "y", x.dtype, (batch, dim), dev)
    with torch.cuda.device(dev):
        st = _stream_handle(stream, dev)
        rc = lib.mamba_state_update(batch, dim, N, io, sp, args[0], args[1], args[2], args[3],
                                    args[4], args[5], args[6], args[7], yp, st)
    if rc != 0:
        raise MambaError(rc, "mamba_state_update")
    return y


def mamba_state_update_ex(state, x, delta, dt_bias, A, B, C, D_skip, z, softplus: bool = True,
                          zoh: bool = False, y=None, stream=None):
    """mamba_state_update with the softplus and zero-order-hold switches."""
    torch = _torch()
    lib = load()
    batch, dim, N = state.shape
    dev = state.device
    io = _io_dtype(x)
    if y is None:
        y = torch.empty_like(x)
    sp = _ptr(state, "state", torch.float32, (batch, dim, N), dev)
    args = (
        _ptr(x, "x", x.dtype, (batch, dim), dev),
        _ptr(delta, "delta", x.dtype, (batch, dim), dev),
        _ptr(dt_bias, "dt_bias", torch.float32, (dim,), dev),
        _ptr(A, "A", torch.float32, (dim, N), dev),
        _ptr(B, "B", x.dtype, (batch, N), dev),
        _ptr(C, "C", x.dtype, (batch, N), dev),
        _ptr(D_skip, "D_skip", torch.float32, (dim,), dev),
        _ptr(z, "z", x.dtype, (batch, dim), dev),
    )
    yp = _ptr(y, "y", x.dtype, (batch, dim), dev)
    with torch.cuda.device(dev):
        st = _stream_handle(stream, dev)
        rc = lib.mamba_state_update_ex(batch, dim, N, io, sp, args[0], args[1], args[2], args[3],
                                       args[4], args[5], args[6], args[7],
                                       scan_flags(softplus, zoh), yp, st)
    if rc != 0:
        raise MambaError(rc, "mamba_state_update_ex")
    return y


def mamba_device_status(stream=None) -> int:
    """Synchronise the stream and read/clear the device error word (0 = ok)."""
    torch = _torch()
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device())
    return lib.mamba_device_status(_stream_handle(stream, dev))


def mamba_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the bounded-wait self-test (a wait that can only time out)."""
    torch = _torch()
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device())
    rc = lib.mamba_selftest_wait_timeout(int(limit_us), _stream_handle(stream, dev))
    if rc != 0:
        raise MambaError(rc, "mamba_selftest_wait_timeout")


def mamba_scan_set_tuning(tail: int = 0, stages: int = 0, chunks: int = 0,
                          layout: int = 0) -> None:
    rc = load().mamba_scan_set_tuning(int(tail), int(stages), int(chunks), int(layout))
    if rc != 0:
        raise MambaError(rc, "mamba_scan_set_tuning")


def mamba_probe_pipe_rate(kind: int, warps_per_subpartition: int, chains: int,
                          iters: int = 4096, stream=None):
    """Measurement support (not part of the scan): sustained lane operations
    per SM clock of one kind of arithmetic; returns (rate, median CTA cycles)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device())
    rate = ctypes.c_double(0.0)
    cyc = ctypes.c_double(0.0)
    rc = load().mamba_probe_pipe_rate(int(kind), int(warps_per_subpartition), int(chains),
                                      int(iters), ctypes.byref(rate), ctypes.byref(cyc),
                                      _stream_handle(stream, dev))
    if rc != 0:
        raise MambaError(rc, "mamba_probe_pipe_rate")
    return rate.value, cyc.value


def mamba_debug_build():
    """(is this the debug build, source line of the last failed index check
    reported by mamba_device_status or 0)."""
    line = ctypes.c_int(0)
    flag = load().mamba_debug_build(ctypes.byref(line))
    return bool(flag), line.value


def mamba_selftest_bounds(stream=None) -> None:
    """Launch the index-check self-test (see include/mamba_scan.h)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device())
    rc = load().mamba_selftest_bounds(_stream_handle(stream, dev))
    if rc != 0:
        raise MambaError(rc, "mamba_selftest_bounds")


def mamba_profile_begin() -> None:
    rc = load().mamba_profile_begin()
    if rc != 0:
        raise MambaError(rc, "mamba_profile_begin")


def mamba_profile_end() -> dict:
    """Stop per-launch timing; return {kind: (total_ms, launches)}."""
    n = len(KIND_NAMES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    rc = load().mamba_profile_end(ms, cnt, n)
    if rc != 0:
        raise MambaError(rc, "mamba_profile_end")
    return {KIND_NAMES[i]: (ms[i], cnt[i]) for i in range(n)}
