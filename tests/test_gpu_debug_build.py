"""The debug build (libmamba_scan_debug.so, compiled with -DMAMBA_DEBUG):
every global load and store of the scan, generation-step, packing, carry,
convolution and backward kernels checks its index against its buffer's extent and,
instead of faulting, skips the access and reports MAMBA_ERR_BOUNDS through
mamba_device_status.  The check runs in a fresh process that loads the debug
library (MAMBA_SCAN_LIBRARY=debug): the odd scan shapes of the parity tests
(tensor-map and element-wise paths, ragged tails), a chunked plan, the
extended modes, both generation-step kernels, the convolution, the backward
pass and the training pair must match the oracle with no failed check, and the index-check self-test must be
reported with its source line."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_passes_every_index_check():
    env = dict(os.environ, MAMBA_SCAN_LIBRARY="debug")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_check.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug build ok" in r.stdout
