"""Seeded synthetic inputs for the selective scan (S6) and its decode update.

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the scan's arithmetic, so both the fp64 oracle (``oracle/``)
and the CUDA library can be fed from it without sharing any method code.

Shapes and value distributions follow the Mamba layer shapes used throughout
("Mamba: linear-time sequence modeling with selective state spaces",
"What they did": the D x N state with N = 16 in the language models, the
block's expansion E = 2, and the S6 parameters u, delta, B, C, z):

* u, z           (batch, D, L)  ~ N(0, 1)
* delta          (batch, D, L)  ~ 0.5 * N(0, 1)   (the pre-softplus input)
* B, C           (batch, N, L)  ~ N(0, 1)
* A              (D, N)         = -(n + 1)        (S4D-real initialisation)
* dt_bias        (D,)           ~ U(lo, hi)       (U(-4,-2), or U(-6,-4) for
                                                   the long-memory case)
* D_skip         (D,)           ~ N(0, 1)

Random streams: numpy's PCG64 bit generator, one independent stream per
(seed, tensor name[, decode step]) built with ``SeedSequence``.  bf16 values
are produced by round-to-nearest-even of the fp32 draw and are stored as
their raw uint16 bit patterns; ``widen`` turns them back into exact fp32/fp64.
"""

from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"


# --------------------------------------------------------------------------
# bf16 storage helpers (bit manipulation only)
# --------------------------------------------------------------------------

def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    # round-to-nearest-even on the 16 dropped bits
    lsb = (bits >> np.uint32(16)) & np.uint32(1)
    rounded = bits + np.uint32(0x7FFF) + lsb
    out = (rounded >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def widen(arr: np.ndarray, dtype: str, to=np.float64) -> np.ndarray:
    """Exact widening of a stored tensor (fp32 values or bf16 bits)."""
    if arr is None:
        return None
    if dtype == BF16 and arr.dtype == np.uint16:
        return bf16_to_f32(arr).astype(to)
    return np.asarray(arr, dtype=np.float32).astype(to)


def to_torch(arr, dtype: str, device="cuda"):
    """Storage-form array (fp32 values or bf16 bits) -> torch tensor on `device`."""
    if arr is None:
        return None
    import torch
    if dtype == BF16 and arr.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    return t.to(device)


def store(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round an fp32 array to the storage dtype (fp32 values or bf16 bits)."""
    if dtype == BF16:
        return bf16_round(x)
    return np.ascontiguousarray(x, dtype=np.float32)


# --------------------------------------------------------------------------
# streams
# --------------------------------------------------------------------------

def _rng(seed: int, name: str, *extra: int) -> np.random.Generator:
    key = [int(seed), zlib.crc32(name.encode())] + [int(e) for e in extra]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


def normal(seed: int, name: str, shape, scale: float = 1.0, *extra: int) -> np.ndarray:
    g = _rng(seed, name, *extra)
    out = g.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        out *= np.float32(scale)
    return out


def uniform(seed: int, name: str, shape, lo: float, hi: float, *extra: int) -> np.ndarray:
    g = _rng(seed, name, *extra)
    return g.uniform(lo, hi, size=shape).astype(np.float32)


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class ScanShape:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    dtype: str = BF16
    dt_lo: float = -4.0
    dt_hi: float = -2.0
    delta_scale: float = 0.5
    softplus: bool = True
    gate: bool = True
    seed: int = 1000
    # u, delta and z drawn from one stream per (tensor, batch entry, channel)
    # instead of one per tensor: any row can be regenerated alone, so
    # sequences of a million steps need neither a full host copy nor a
    # transfer back from the device to check sampled rows
    rowwise: bool = False

    @property
    def elems(self) -> int:
        return self.batch * self.dim * self.seqlen

    def io_bytes(self) -> int:
        """Bytes of u, delta, z, y (batch*D*L each) and B, C (batch*N*L each)."""
        es = 2 if self.dtype == BF16 else 4
        big = 4 if self.gate else 3
        return es * (big * self.batch * self.dim * self.seqlen
                     + 2 * self.batch * self.dstate * self.seqlen)


@dataclasses.dataclass(frozen=True)
class DecodeShape:
    name: str
    batch: int
    dim: int
    dstate: int
    steps: int
    dtype: str = BF16
    dt_lo: float = -4.0
    dt_hi: float = -2.0
    delta_scale: float = 0.5
    seed: int = 1004

    def io_bytes_per_step(self) -> int:
        """x, delta, z, y (batch*D each) and B, C (batch*N each), storage dtype."""
        es = 2 if self.dtype == BF16 else 4
        return es * (4 * self.batch * self.dim + 2 * self.batch * self.dstate)

    def state_bytes(self) -> int:
        return 4 * self.batch * self.dim * self.dstate


# The five workloads: a tiny fp32 case, the Mamba-130M and Mamba-2.8B layer
# shapes (d_model 768 / 2560, E = 2), a 262144-token single-sequence scan and
# a 1024-step batched decode on the 2.8B layer shape.
TINY = ScanShape("tiny-fp32 b1 d16 n4 l64", 1, 16, 4, 64, dtype=F32, seed=1000)
M130 = ScanShape("mamba130m-layer b8 d1536 n16 l2048", 8, 1536, 16, 2048, seed=1001)
M2P8 = ScanShape("mamba2.8b-layer b4 d5120 n16 l2048", 4, 5120, 16, 2048, seed=1002)
LONG = ScanShape("long b1 d1536 n16 l262144", 1, 1536, 16, 262144,
                 dt_lo=-6.0, dt_hi=-4.0, seed=1003)
DECODE = DecodeShape("decode b128 d5120 n16 x1024", 128, 5120, 16, 1024, seed=1004)

# the length the induction-head result on the pages extrapolates to
LONG1M = ScanShape("long1m b1 d1536 n16 l1048576", 1, 1536, 16, 1 << 20,
                   dt_lo=-6.0, dt_hi=-4.0, seed=1005, rowwise=True)

SCAN_SHAPES = {"tiny": TINY, "m130": M130, "m2p8": M2P8, "long": LONG, "long1m": LONG1M}


def s4d_real_A(dim: int, dstate: int) -> np.ndarray:
    """A[d, n] = -(n + 1): the real diagonal initialisation used by the configs."""
    return np.tile(-(np.arange(dstate, dtype=np.float32) + 1.0), (dim, 1))


def scan_inputs(shape: ScanShape, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """All inputs of one scan call in storage form.

    Keys: u, delta, z, B, C (storage dtype: fp32 values or bf16 bits),
    A, dt_bias, D_skip (fp32), plus 'dtype' and 'softplus'.
    """
    s = shape.seed if seed is None else seed
    bt, d, n, l = shape.batch, shape.dim, shape.dstate, shape.seqlen
    if shape.rowwise:
        out = rowwise_small_inputs(shape, seed)
        for k in ("u", "delta", "z"):
            out[k] = np.stack([rows_block(shape, k, b, 0, d, seed) for b in range(bt)])
        return out
    out = {
        "u": store(normal(s, "u", (bt, d, l)), shape.dtype),
        "delta": store(normal(s, "delta", (bt, d, l), shape.delta_scale), shape.dtype),
        "z": store(normal(s, "z", (bt, d, l)), shape.dtype) if shape.gate else None,
        "B": store(normal(s, "B", (bt, n, l)), shape.dtype),
        "C": store(normal(s, "C", (bt, n, l)), shape.dtype),
        "A": s4d_real_A(d, n),
        "dt_bias": uniform(s, "dt_bias", (d,), shape.dt_lo, shape.dt_hi),
        "D_skip": normal(s, "D_skip", (d,)),
    }
    out["dtype"] = shape.dtype
    out["softplus"] = shape.softplus
    return out


def rows_block(shape: ScanShape, name: str, b: int, d0: int, d1: int,
               seed: Optional[int] = None) -> np.ndarray:
    """Storage-form rows [d0, d1) of batch entry b of tensor `name` (u, delta
    or z) of a row-wise shape, shape (d1 - d0, L): row (b, d) comes from its
    own stream keyed by (seed, name, b, d)."""
    assert shape.rowwise
    s = shape.seed if seed is None else seed
    scale = shape.delta_scale if name == "delta" else 1.0
    out = np.empty((d1 - d0, shape.seqlen), np.float32)
    for i, d in enumerate(range(d0, d1)):
        out[i] = normal(s, name, (shape.seqlen,), scale, b, d)
    return store(out, shape.dtype)


def rowwise_to_device(shape: ScanShape, name: str, device="cuda", seed: Optional[int] = None,
                      block_rows: int = 32, threads: Optional[int] = None):
    """Tensor `name` (u, delta or z) of a row-wise shape as a torch tensor on
    `device`, generated in blocks of rows by a pool of host threads (numpy's
    generators release the GIL) and copied block by block, so that no full
    host copy is ever held."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    import torch
    tdt = torch.bfloat16 if shape.dtype == BF16 else torch.float32
    out = torch.empty((shape.batch, shape.dim, shape.seqlen), dtype=tdt, device=device)
    jobs = [(b, d0, min(shape.dim, d0 + block_rows))
            for b in range(shape.batch) for d0 in range(0, shape.dim, block_rows)]
    nthr = threads or min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=nthr) as pool:
        for (b, d0, d1), blk in zip(jobs, pool.map(
                lambda j: rows_block(shape, name, j[0], j[1], j[2], seed), jobs)):
            out[b, d0:d1].copy_(to_torch(blk, shape.dtype, "cpu"))
    return out


def rowwise_small_inputs(shape: ScanShape, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """The inputs of a row-wise shape other than u, delta and z: B, C, A,
    dt_bias, D_skip (storage form / fp32), plus 'dtype' and 'softplus'."""
    assert shape.rowwise
    s = shape.seed if seed is None else seed
    bt, d, n, l = shape.batch, shape.dim, shape.dstate, shape.seqlen
    return {"B": store(normal(s, "B", (bt, n, l)), shape.dtype),
            "C": store(normal(s, "C", (bt, n, l)), shape.dtype),
            "A": s4d_real_A(d, n),
            "dt_bias": uniform(s, "dt_bias", (d,), shape.dt_lo, shape.dt_hi),
            "D_skip": normal(s, "D_skip", (d,)),
            "dtype": shape.dtype, "softplus": shape.softplus}


def rowwise_sample(shape: ScanShape, rows, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """The sampled rows (flat b*D + d indices, all of one batch entry) of a
    row-wise shape as a problem of its own: batch 1, one channel per sampled
    row, in the layout of scan_inputs (u, delta, z (1, R, L); B, C (1, N, L);
    A (R, N); dt_bias, D_skip (R,))."""
    small = rowwise_small_inputs(shape, seed)
    rows = np.asarray(rows, np.int64)
    bs, ds = rows // shape.dim, rows % shape.dim
    assert np.all(bs == bs[0]), "rows of one batch entry"
    b = int(bs[0])
    out = {k: np.stack([rows_block(shape, k, b, int(d), int(d) + 1, seed)[0] for d in ds])[None]
           for k in ("u", "delta", "z")}
    out.update(B=small["B"][b:b + 1], C=small["C"][b:b + 1], A=small["A"][ds],
               dt_bias=small["dt_bias"][ds], D_skip=small["D_skip"][ds],
               dtype=shape.dtype, softplus=shape.softplus)
    return out


def decode_params(shape: DecodeShape, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Per-channel parameters of the decode workload (fp32)."""
    s = shape.seed if seed is None else seed
    return {
        "A": s4d_real_A(shape.dim, shape.dstate),
        "dt_bias": uniform(s, "dt_bias", (shape.dim,), shape.dt_lo, shape.dt_hi),
        "D_skip": normal(s, "D_skip", (shape.dim,)),
    }


def decode_step_inputs(shape: DecodeShape, step: int, seed: Optional[int] = None,
                       rows: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Fresh x, delta, z (batch, D) and B, C (batch, N) for one decode step."""
    s = shape.seed if seed is None else seed
    bt, d, n = shape.batch, shape.dim, shape.dstate
    out = {
        "x": store(normal(s, "x", (bt, d), 1.0, step), shape.dtype),
        "delta": store(normal(s, "delta", (bt, d), shape.delta_scale, step), shape.dtype),
        "z": store(normal(s, "z", (bt, d), 1.0, step), shape.dtype),
        "B": store(normal(s, "B", (bt, n), 1.0, step), shape.dtype),
        "C": store(normal(s, "C", (bt, n), 1.0, step), shape.dtype),
    }
    out["dtype"] = shape.dtype
    return out


def sample_rows(seed: int, batch: int, dim: int, count: int) -> np.ndarray:
    """A fixed, seeded sample of distinct (b, d) rows, as flat indices b*dim + d."""
    g = _rng(seed, "rows")
    count = min(count, batch * dim)
    return np.sort(g.choice(batch * dim, size=count, replace=False)).astype(np.int64)
