"""Selective scan (S6) and single-token state update on B300 (sm_103a).

Thin Python binding over the C ABI in ``include/mamba_scan.h``
(``libmamba_scan.so``, built in-tree by ``build.py``).  The functions keep the
C names and argument order; they only check tensor properties, pass device
pointers and the current CUDA stream, and turn status codes into exceptions.
Every step of the computation runs in the library's CUDA kernels: there is
no CPU or PyTorch fallback, and calling without the built library raises.
"""

from .autograd import mamba_scan_fn  # noqa: F401
from ._lib import (  # noqa: F401
    KIND_NAMES,
    MAMBA_BF16,
    MAMBA_F32,
    MAMBA_FLAG_NOALLOC,
    MAMBA_FLAG_SOFTPLUS,
    MAMBA_FLAG_ZOH,
    MambaError,
    checkpoint_shape,
    lib_path,
    load,
    mamba_conv1d_fwd,
    mamba_conv1d_update,
    mamba_debug_build,
    mamba_device_status,
    mamba_profile_begin,
    mamba_probe_pipe_rate,
    mamba_profile_end,
    mamba_scan_bwd,
    mamba_scan_bwd_ckpt,
    mamba_scan_checkpoint_bytes,
    mamba_scan_fwd,
    mamba_scan_fwd_ex,
    mamba_scan_fwd_noalloc,
    mamba_scan_fwd_train,
    mamba_scan_set_tuning,
    mamba_selftest_bounds,
    mamba_selftest_wait_timeout,
    mamba_state_update,
    mamba_state_update_ex,
    mamba_status_string,
    mamba_version,
)
