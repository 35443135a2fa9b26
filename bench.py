#!/usr/bin/env python3
"""Benchmark of the selective scan (S6) forward on one GPU per process.

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]

One step = one mamba_scan_fwd call over the Mamba-2.8B layer workload
(batch 4, D 5120, N 16, L 2048, bf16 u/delta/z/B/C/y, fp32 A/dt_bias/D_skip,
fp32 final state written), i.e. every stage of the scan path: Delta/softplus,
discretisation, the time recurrence, the chunk carry when the plan uses one,
skip term, silu gate and the final state.  Inputs (336 MB) are larger than
the 126 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  value = B*L*D elements per second summed over
all ranks (each rank scans its own independently seeded batch: weak scaling).
The line carries the roofline of the dominant kernel (timed per launch with
CUDA events on its stream), an end-to-end figure through pinned host memory,
SM clocks sampled during the timed region, the decode step, and the fp64 CPU
oracle timed on a bounded sample of the same workload.  Further objects time,
on the same inputs, the extended scan (initial state; Euler and zero-order
hold), the backward pass and the causal convolution with its generation
step (--no-ext, --no-bwd, --no-conv skip them).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "scan throughput (B*L*D elems/s)"
UNIT = "elems/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "scan_traffic.json")
# the output of `python bench.py --pipe-rates` on a B300 (measured per-SM
# rates of the scan's arithmetic), the source of the measured ceiling
PIPE_RATES_FILE = os.path.join(ROOT, "profiles", "pipe_rates.json")
KERNEL_SRC = os.path.join(ROOT, "selective_state_space_135_b300", "csrc", "mamba_scan.cu")
# Per-SM unit counts of B300 (sm_103): 128 fp32 lanes (one fp32 multiply or
# FMA per lane per clock, packed f32x2 included) and 32 ex2 results per clock
# on the special-function units; 148 SMs.  One state update of the scan
# (one (b, d, t, n) element) needs 4 fp32 lane operations (Delta*A, Delta*u*B,
# the state FMA, the C.h FMA) and one ex2, so both units give the same peak:
# 148 * 32 * f_sm state updates per second.
FP32_LANES_PER_SM = 128
FP32_OPS_PER_UPDATE = 4
EX2_PER_CLK_SM = 32
N_SM = 148
FALLBACK_HBM_GBS = 6400.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------------------
# environment

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "sm_max_mhz": 2032.0}, "fallback"


def kernel_hash():
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_traffic(workload_name):
    """DRAM bytes per launch of the scan kernel from a committed ncu summary,
    only if it was taken on the current kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        if t.get("kernel_sha256_16") == kernel_hash() and t.get("workload") == workload_name:
            return float(t["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# --------------------------------------------------------------------------
# multi-rank bookkeeping (weak scaling: every rank scans its own batch)

def rank_seed(shape, rank):
    """Seed of rank `rank`'s independent copy of the workload."""
    return shape.seed + 7919 * rank


def max_over_ranks(x, dist_mod=None, device=None):
    """The largest value of `x` over all ranks (x itself on one rank)."""
    if dist_mod is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(elems_per_step, steps, world, ms):
    """Elements per second summed over all ranks, timed by the slowest rank."""
    return elems_per_step * steps * world / (ms * 1e-3)


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                     power=float(parts[3]) if parts[3] not in ("[N/A]", "") else None,
                                     hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
            if any(r[key] == "Active" for r in rows):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "samples": len(rows),
                "power_w_max": max((r["power"] for r in rows if r["power"] is not None),
                                   default=None),
                "reasons": reasons}


# --------------------------------------------------------------------------
# CPU oracle leg (also the reference arm)

def oracle_on_rows(inp, shape, rows):
    """Seconds the fp64 oracle, as it stands, takes to scan the given (b, d)
    rows of the workload (inputs drawn before the clock starts)."""
    import oracle
    if inp is not None:
        t0 = time.perf_counter()
        oracle.scan_rows(inp, rows)
        return time.perf_counter() - t0
    # row-wise workload (one batch entry): the sampled rows as one problem
    w = oracle.scan_inputs_f64(synth.rowwise_sample(shape, rows))
    t0 = time.perf_counter()
    oracle.scan(w["u"], w["delta"], w["A"], w["B"], w["C"], dt_bias=w["dt_bias"],
                D_skip=w["D_skip"], z=w["z"])
    return time.perf_counter() - t0


def oracle_on_channels(inp, chs, threads=None):
    """Seconds the fp64 oracle, as it stands, takes to scan every batch entry
    of the channels `chs` in one call (batch x len(chs) rows, which the
    oracle spreads over its threads; inputs widened before the clock
    starts), and the threads it used."""
    import oracle
    dt = inp["dtype"]
    zs = inp.get("z")
    u = synth.widen(inp["u"][:, chs], dt)
    dl = synth.widen(inp["delta"][:, chs], dt)
    z = None if zs is None else synth.widen(zs[:, chs], dt)
    Bw, Cw = synth.widen(inp["B"], dt), synth.widen(inp["C"], dt)
    A = np.asarray(inp["A"], np.float64)[chs]
    dtb = np.asarray(inp["dt_bias"], np.float64)[chs]
    dsk = np.asarray(inp["D_skip"], np.float64)[chs]
    t0 = time.perf_counter()
    _, _, used = oracle.scan(u, dl, A, Bw, Cw, dt_bias=dtb, D_skip=dsk, z=z, threads=threads)
    return time.perf_counter() - t0, used


def _sample_channels(shape, n, seed):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(shape.dim, size=int(max(1, min(n, shape.dim))), replace=False))


def _oracle_channels_for(inp, shape, seconds, seed, threads=None):
    """Channels of `shape` (all batch entries each) the oracle scans in about
    `seconds`."""
    ncores = threads or os.cpu_count() or 1
    k0 = max(2, 4 * -(-ncores // shape.batch))   # several rows for every thread
    secs, _ = oracle_on_channels(inp, _sample_channels(shape, k0, seed), threads)
    per_ch = max(secs, 1e-4) / k0
    return int(max(1, min(shape.dim, seconds / per_ch)))


def _oracle_rows_for(inp, shape, seconds, seed):
    """Rows of `shape` the oracle scans in about `seconds` on all host cores."""
    ncores = os.cpu_count() or 1
    probe = synth.sample_rows(seed, shape.batch, shape.dim, min(ncores, 64))
    slot = max(oracle_on_rows(inp, shape, probe), 1e-3) / len(probe) * min(ncores, len(probe))
    return int(max(1, min(shape.batch * shape.dim, seconds / slot * ncores)))


def oracle_rate(inp, shape, target_s):
    """Time the fp64 oracle, as it stands, on a seeded sample of rows: whole
    channels (every batch entry) of an in-memory workload, sampled rows of a
    row-wise one.  Returns (elems/s, threads, rows, seconds)."""
    if inp is not None:
        n_ch = _oracle_channels_for(inp, shape, target_s, 1234)
        secs, used = oracle_on_channels(inp, _sample_channels(shape, n_ch, 1235))
        nrows = shape.batch * n_ch
        return nrows * shape.seqlen / secs, used, nrows, secs
    nrows = _oracle_rows_for(inp, shape, target_s, 1234)
    rows = synth.sample_rows(1235, shape.batch, shape.dim, nrows)
    secs = oracle_on_rows(inp, shape, rows)
    threads = min(os.cpu_count() or 1, len(rows))
    return len(rows) * shape.seqlen / secs, threads, len(rows), secs


def oracle_single_core(seconds):
    """The fp64 oracle, as it stands, on one host thread: a seeded sample of
    full-length rows of the Mamba-130M layer workload (B8 D1536 N16 L2048),
    about `seconds` of work.  Returns the cpu_baseline-style object."""
    import oracle
    shape = synth.M130
    inp = synth.scan_inputs(shape)
    probe = synth.sample_rows(77, shape.batch, shape.dim, 4)
    t0 = time.perf_counter()
    oracle.scan_rows(inp, probe, threads=1)
    per_row = max(time.perf_counter() - t0, 1e-4) / len(probe)
    n = int(max(1, min(shape.batch * shape.dim, seconds / per_row)))
    rows = synth.sample_rows(78, shape.batch, shape.dim, n)
    t0 = time.perf_counter()
    oracle.scan_rows(inp, rows, threads=1)
    secs = time.perf_counter() - t0
    return {"value": n * shape.seqlen / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} seeded (b,d) rows of {shape.name}, full length {shape.seqlen}, "
                      f"N={shape.dstate}; {secs:.1f} s on 1 thread"}


def config_dict(shape, ws):
    return {"workload": shape.name, "batch": shape.batch, "dim": shape.dim,
            "dstate": shape.dstate, "seqlen": shape.seqlen, "io_dtype": shape.dtype,
            "state_dtype": "f32", "gate": "silu(z)", "softplus": True, "final_state": True,
            "l2": f"inputs {shape.io_bytes() / 1e6:.0f} MB > 126 MB L2, no flush",
            "parallelism": f"{ws} independent replica(s), one batch per GPU"}


def run_reference(args, shape):
    """The reference arm: the fp64 CPU oracle, as it stands, on host cores."""
    import oracle
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp = None if shape.rowwise else synth.scan_inputs(shape)
    per_step = max(0.2, 150.0 / max(1, args.steps + args.warmup))
    if inp is not None:   # whole channels, every batch entry, in one oracle call
        n_ch = _oracle_channels_for(inp, shape, per_step, 99)
        chs = _sample_channels(shape, n_ch, 100)
        for _ in range(args.warmup):
            oracle_on_channels(inp, chs)
        runs = [oracle_on_channels(inp, chs) for _ in range(args.steps)]
        secs = sum(r[0] for r in runs)
        threads = max(r[1] for r in runs)
        nrows = shape.batch * n_ch
        sample = (f"{nrows} (b,d) rows per step ({n_ch} seeded channels x all {shape.batch} "
                  f"batch entries) of the {shape.name} workload, full length {shape.seqlen}, "
                  f"N={shape.dstate}")
    else:
        nrows = _oracle_rows_for(inp, shape, per_step, 99)
        rows = synth.sample_rows(100, shape.batch, shape.dim, nrows)
        for _ in range(args.warmup):
            oracle_on_rows(inp, shape, rows)
        secs = sum(oracle_on_rows(inp, shape, rows) for _ in range(args.steps))
        threads = min(os.cpu_count() or 1, nrows)
        sample = (f"{nrows} seeded (b,d) rows of the {shape.name} workload per step, full "
                  f"length {shape.seqlen}, N={shape.dstate}")
    value = nrows * shape.seqlen * args.steps / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(shape, ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# arithmetic rates (the denominators of the scan's roofline)

PIPE_KINDS = {0: "ex2", 1: "lg2", 2: "tanh", 3: "ffma2 (lane-ops)", 4: "ffma",
              5: "scan state update (2 ex2 + 4 packed ops per 2 updates)"}


def load_pipe_ceiling():
    """State updates per clock per SM that the scan's core arithmetic reaches
    alone on B300 (committed measurement), or None."""
    try:
        with open(PIPE_RATES_FILE) as f:
            return float(json.load(f)["scan_core_ceiling"]["state_updates_per_clk_sm"])
    except Exception:
        return None


def run_pipe_rates():
    """Sustained per-SM rates, in lane operations per SM clock, of each kind
    of arithmetic the scan uses, with 1 to 8 warps per SM sub-partition and
    8 or 16 independent chains per thread (1 to 16 for the scan's state
    update, whose chains are the state pairs a thread holds) (the library's
    mamba_probe_pipe_rate, clock64 inside the kernel)."""
    import torch
    import selective_state_space_135_b300 as mm
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    torch.cuda.set_device(0)
    rows = []
    for kind in sorted(PIPE_KINDS):
        for wps in (1, 2, 3, 4, 5, 8):
            for chains in (1, 2, 4, 8, 16):
                if kind != 5 and chains not in (8, 16):
                    continue
                try:
                    rate, cyc = mm.mamba_probe_pipe_rate(kind, wps, chains, iters=4096)
                except mm.MambaError:
                    continue   # more registers than the SM has at this warp count
                rows.append({"kind": PIPE_KINDS[kind], "warps_per_subpartition": wps,
                             "chains": chains, "ops_per_clk_sm": round(rate, 3),
                             "cycles": int(cyc)})
    peaks, src = load_peaks()
    smax = float(peaks.get("sm_max_mhz", 2032.0))
    best = {}
    for r in rows:
        best[r["kind"]] = max(best.get(r["kind"], 0.0), r["ops_per_clk_sm"])
    scan = best[PIPE_KINDS[5]]
    print(json.dumps({
        "pipe_rates": rows, "best_ops_per_clk_sm": best,
        "scan_core_ceiling": {
            "state_updates_per_clk_sm": scan,
            "T_updates_per_s": scan * N_SM * smax * 1e6 / 1e12,
            "m2p8_us": synth.M2P8.batch * synth.M2P8.dim * synth.M2P8.seqlen * synth.M2P8.dstate
                       / (scan * N_SM * smax * 1e6) * 1e6,
            "at_mhz": smax, "sm_count": N_SM},
    }), flush=True)
    return 0


# --------------------------------------------------------------------------
# our arm

def run_ours(args, shape):
    import torch
    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the scan has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    import selective_state_space_135_b300 as mm
    mm.mamba_scan_set_tuning(0, 0, 0, args.layout)

    seed = rank_seed(shape, rank)
    dt = shape.dtype
    if shape.rowwise:
        # row-wise streams: generated block by block straight into device
        # memory (the host never holds a full tensor)
        inp = None
        small = synth.rowwise_small_inputs(shape, seed=seed)
        u, delta, z = (synth.rowwise_to_device(shape, k, dev, seed=seed)
                       for k in ("u", "delta", "z"))
        B, C = (synth.to_torch(small[k], dt, dev) for k in ("B", "C"))
        src = small
    else:
        inp = synth.scan_inputs(shape, seed=seed)
        u, delta, z, B, C = (synth.to_torch(inp[k], dt, dev) for k in ("u", "delta", "z", "B", "C"))
        src = inp
    A = torch.from_numpy(src["A"]).to(dev)
    dtb = torch.from_numpy(src["dt_bias"]).to(dev)
    dsk = torch.from_numpy(src["D_skip"]).to(dev)
    y = torch.empty_like(u)
    fin = torch.empty((shape.batch, shape.dim, shape.dstate), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        mm.mamba_scan_fwd(u, delta, dtb, A, B, C, dsk, z, True, y=y, final_state=fin,
                          stream=stream)

    def barrier():
        if pg:
            pg.barrier()
        torch.cuda.synchronize(dev)

    # bring clocks to steady state, then sample them through warm-up and timing
    sampler = ClockSampler(local)
    sampler.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        for _ in range(50):
            step()
        torch.cuda.synchronize(dev)
    for _ in range(args.warmup):
        step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    mm.mamba_profile_begin()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    prof = mm.mamba_profile_end()
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), pg, dev)
    value = whole_job_rate(shape.elems, args.steps, ws, ms)
    ms_per_step = ms / args.steps

    # The roofline is taken over the whole scan call: its main pass may run
    # as two overlapping launches (whole-sequence units on the caller's
    # stream, the chunked tail on the library's side stream), so the per-call
    # time measured by the CUDA events around the timed steps is the time of
    # the dominant work.  Per-launch averages by kernel kind are kept as
    # context.
    launches = sum(n for _, n in prof.values())
    k_ms = ms_per_step
    peaks, peak_src = load_peaks()
    smax = float(peaks.get("sm_max_mhz", 2032.0))
    updates = shape.batch * shape.dim * shape.seqlen * shape.dstate
    alu_peak = min(FP32_LANES_PER_SM / FP32_OPS_PER_UPDATE, EX2_PER_CLK_SM) * N_SM * smax * 1e6
    alu_achieved = updates / (k_ms * 1e-3)
    ceiling = load_pipe_ceiling()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    hbm_achieved = shape.io_bytes() / (k_ms * 1e-3) / 1e9
    traffic = load_traffic(shape.name)
    roofline = {
        "bound": "alu",
        "achieved": alu_achieved / 1e12, "peak": alu_peak / 1e12, "unit": "T state-updates/s",
        "frac": alu_achieved / alu_peak, "traffic": traffic,
        "kernel": "mamba_scan_fwd call (B/C pack + main passes)", "kernel_ms": k_ms,
        "launch_ms_by_kind": {k: v[0] / v[1] for k, v in prof.items() if v[1]},
        "peak_source": f"{N_SM} SMs x min({FP32_LANES_PER_SM} fp32 lanes / "
                       f"{FP32_OPS_PER_UPDATE} ops, {EX2_PER_CLK_SM} ex2) per clock x "
                       f"{smax:.0f} MHz ({peak_src} sm_max)",
        "work_per_launch": f"{updates:.4g} state updates (B*D*L*N)",
        "measured_ceiling": None if ceiling is None else {
            "achieved": alu_achieved / 1e12,
            "peak": ceiling * N_SM * smax * 1e6 / 1e12, "unit": "T state-updates/s",
            "frac": alu_achieved / (ceiling * N_SM * smax * 1e6),
            "peak_source": f"{ceiling:.2f} state updates per clock per SM (the state update's "
                           f"2 ex2 + 4 packed fp32 ops, measured alone: profiles/pipe_rates.json)"
                           f" x {N_SM} SMs x {smax:.0f} MHz"},
        "hbm": {"achieved": hbm_achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": hbm_achieved / hbm_peak, "peak_source": peak_src,
                "algorithmic_bytes_per_launch": shape.io_bytes(),
                "traffic_per_launch": traffic},
    }

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_dict(shape, ws),
        "roofline": roofline,
        "gpu_launches": launches,
        "launches_by_kernel": {k: v[1] for k, v in prof.items()},
        "clocks": clocks,
    }

    if not args.no_e2e and inp is not None:
        line["e2e"] = e2e_leg(args, shape, inp, dev, stream, mm, ws, pg)
    if not args.no_decode and rank == 0:
        line["decode"] = decode_leg(dev, mm)
    if not args.no_ext and rank == 0:
        line["ext"] = ext_leg(shape, (u, delta, dtb, A, B, C, dsk, z), y, fin, dev, stream, mm)
    if not args.no_bwd and rank == 0:
        line["bwd"] = bwd_leg(shape, (u, delta, dtb, A, B, C, dsk, z), dev, stream, mm)
    if not args.no_conv and rank == 0:
        line["conv"] = conv_leg(shape, u, dev, stream, mm)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, thr, nrows, secs = oracle_rate(inp, shape, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": v, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": (f"{nrows} (b,d) rows ({nrows // shape.batch} seeded channels x all "
                       f"{shape.batch} batch entries) of {shape.name}, full length {shape.seqlen}, "
                       f"N={shape.dstate}; {secs:.1f} s on {thr} threads") if inp is not None else
                      (f"{nrows} seeded (b,d) rows of {shape.name}, full length {shape.seqlen}, "
                       f"N={shape.dstate}; {secs:.1f} s on {thr} threads"),
            "single_core_m130": oracle_single_core(args.cpu_seconds / 2)}
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def e2e_leg(args, shape, inp, dev, stream, mm, ws, pg):
    """Same metric through the public call with host buffers: every step copies
    its inputs from pinned host memory and reads y and the final state back,
    as a user streaming batches would.  The copies of neighbouring steps run
    on their own streams (double-buffered device buffers), so step i's scan
    overlaps step i+1's upload and step i-1's download; every copy of every
    timed step is inside the timed region."""
    import torch
    dt = shape.dtype
    names = ("u", "delta", "z", "B", "C")
    host = {k: synth.to_torch(inp[k], dt, "cpu").pin_memory() for k in names}
    devb = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    A = torch.from_numpy(inp["A"]).to(dev)
    dtb = torch.from_numpy(inp["dt_bias"]).to(dev)
    dsk = torch.from_numpy(inp["D_skip"]).to(dev)
    ys = [torch.empty_like(devb[0]["u"]) for _ in range(2)]
    fins = [torch.empty((shape.batch, shape.dim, shape.dstate), dtype=torch.float32, device=dev)
            for _ in range(2)]
    y_h = [torch.empty_like(ys[0], device="cpu").pin_memory() for _ in range(2)]
    f_h = [torch.empty_like(fins[0], device="cpu").pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = ys[0].numel() * ys[0].element_size() + fins[0].numel() * 4
    # One upload and one download stream: the host link, not the copy
    # engines, bounds these copies (two upload streams measured no faster).
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def step(i):
        sl = i % 2
        with torch.cuda.stream(s_in):
            if used[sl]:
                s_in.wait_event(ev_cmp[sl])          # the scan of step i-2 has read them
            for k in names:
                devb[sl][k].copy_(host[k], non_blocking=True)
            ev_in[sl].record(s_in)
        stream.wait_event(ev_in[sl])
        if used[sl]:
            stream.wait_event(ev_out[sl])            # y of step i-2 has been read back
        b = devb[sl]
        mm.mamba_scan_fwd(b["u"], b["delta"], dtb, A, b["B"], b["C"], dsk, b["z"], True,
                          y=ys[sl], final_state=fins[sl], stream=stream)
        ev_cmp[sl].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[sl])
            y_h[sl].copy_(ys[sl], non_blocking=True)
            f_h[sl].copy_(fins[sl], non_blocking=True)
            ev_out[sl].record(s_out)
        used[sl] = True

    k = max(3, min(args.steps, args.e2e_steps))
    for i in range(3):
        step(i)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(k):
        step(3 + i)
    stream.wait_event(ev_out[(3 + k - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), pg, dev)
    return {"value": whole_job_rate(shape.elems, k, ws, ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k,
            "ms_per_step": ms / k, "overlap": "h2d / scan / d2h of neighbouring steps"}


def ext_leg(shape, ins, y, fin, dev, stream, mm, steps=200, warmup=5):
    """The extended entry point on the same workload: Euler and zero-order
    hold, each starting from a (random) initial state, every entry using all
    steps.  Device-resident inputs, CUDA events on the launching stream."""
    import torch
    g = torch.Generator(device=dev).manual_seed(7)
    h0 = 0.3 * torch.randn((shape.batch, shape.dim, shape.dstate), device=dev, generator=g)
    out = {}
    for name, zoh in (("euler_initial_state", False), ("zoh_initial_state", True)):
        def step():
            mm.mamba_scan_fwd_ex(*ins, softplus=True, zoh=zoh, initial_state=h0, y=y,
                                 final_state=fin, stream=stream)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        out[name] = {"ms_per_step": ms, "value": shape.elems / (ms * 1e-3), "unit": UNIT,
                     "steps": steps}
    return out


def bwd_leg(shape, ins, dev, stream, mm, steps=10, warmup=3):
    """The backward pass on the same workload: gradients of every input from
    a random dy, with the final-state gradient off.  Device-resident inputs
    and outputs, CUDA events on the launching stream; per-kind device times
    from the library's launch timing.  Also the training pair: the forward
    that keeps the checkpoints (mamba_scan_fwd_train) and the backward from
    them (mamba_scan_bwd_ckpt), each timed alone, against the plain forward
    and backward."""
    import torch
    g = torch.Generator(device=dev).manual_seed(11)
    dy = torch.randn(ins[0].shape, device=dev, generator=g).to(ins[0].dtype)
    out = mm.mamba_scan_bwd(*ins, dy, stream=stream)

    def timed(fn, n, prof=False):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if prof:
            mm.mamba_profile_begin()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        kinds = mm.mamba_profile_end() if prof else None
        return e0.elapsed_time(e1) / n, kinds

    ms, prof = timed(lambda: mm.mamba_scan_bwd(*ins, dy, out=out, stream=stream), steps, True)
    updates = shape.batch * shape.dim * shape.seqlen * shape.dstate
    res = {"ms_per_step": ms, "value": shape.elems / (ms * 1e-3), "unit": UNIT, "steps": steps,
           "state_updates_per_s": updates / (ms * 1e-3),
           "launch_ms_by_kind": {k: v[0] / v[1] for k, v in prof.items() if v[1]},
           "note": "checkpoint pass + reverse pass (recomputes each 12-step tile) + reductions; "
                   "the checkpoint pass's own scan, chunk-summary and carry launches are also "
                   "listed under their kinds"}
    y = torch.empty_like(ins[0])
    ck = torch.empty(mm.checkpoint_shape(shape.batch, shape.dim, shape.dstate, shape.seqlen),
                     dtype=torch.float32, device=dev)
    fwd_ms, _ = timed(lambda: mm.mamba_scan_fwd(*ins, True, y=y, stream=stream), steps)
    train_ms, _ = timed(lambda: mm.mamba_scan_fwd_train(*ins, True, y=y, checkpoints=ck,
                                                        stream=stream), steps)
    bwd_ck_ms, prof2 = timed(lambda: mm.mamba_scan_bwd_ckpt(*ins, dy, ck, out=out, stream=stream),
                             steps, True)
    res["from_checkpoints"] = {
        "fwd_train_ms": train_ms, "bwd_ckpt_ms": bwd_ck_ms,
        "train_step_ms": train_ms + bwd_ck_ms, "fwd_plus_bwd_ms": fwd_ms + ms,
        "fwd_ms": fwd_ms, "checkpoint_bytes": ck.numel() * 4,
        "bwd_ckpt_launch_ms_by_kind": {k: v[0] / v[1] for k, v in prof2.items() if v[1]},
        "note": "mamba_scan_fwd_train keeps the state every 12 steps; mamba_scan_bwd_ckpt "
                "starts from them (same gradients, bit for bit)"}
    return res


def conv_leg(shape, x, dev, stream, mm, width=4, steps=50, warmup=5):
    """The causal width-4 convolution + SiLU on the workload's input tensor
    (one read of x, one write of the output, plus the carried state), and its
    generation step on the decode workload's (batch, dim).  HBM-bound: the
    roofline is the measured copy bandwidth."""
    import torch
    g = torch.Generator(device=dev).manual_seed(13)
    w = torch.randn((shape.dim, width), device=dev, generator=g) / 2
    bias = torch.randn((shape.dim,), device=dev, generator=g)
    out = torch.empty_like(x)
    fin = torch.empty((shape.batch, shape.dim, width - 1), dtype=x.dtype, device=dev)
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))

    def timed(fn, n):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n

    ms = timed(lambda: mm.mamba_conv1d_fwd(x, w, bias, silu=True, out=out, final_conv_state=fin,
                                           stream=stream), steps)
    nbytes = 2 * x.numel() * x.element_size() + fin.numel() * fin.element_size()
    dshp = synth.DECODE
    xs = torch.randn((dshp.batch, dshp.dim), device=dev, generator=g).to(x.dtype)
    st = torch.zeros((dshp.batch, dshp.dim, width - 1), dtype=x.dtype, device=dev)
    wd = torch.randn((dshp.dim, width), device=dev, generator=g) / 2
    ys = torch.empty_like(xs)
    # the generation step from a captured graph of 200 steps (no launch cost)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(3):
            mm.mamba_conv1d_update(st, xs, wd, None, out=ys, stream=side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(200):
            mm.mamba_conv1d_update(st, xs, wd, None, out=ys, stream=side)
    graph.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    ms_step = e0.elapsed_time(e1) / 200
    step_bytes = 2 * xs.numel() * xs.element_size() + 2 * st.numel() * st.element_size()
    return {"width": width, "ms_per_call": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9,
            "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm, "bytes_per_call": nbytes,
            "step_us": ms_step * 1e3, "step_GB/s": step_bytes / (ms_step * 1e-3) / 1e9,
            "step_workload": f"decode b{dshp.batch} d{dshp.dim}", "peak_source": src}


def l2_copy_rate(dev, mib=24, reps=400):
    """GB/s (read + write) of a device copy whose source and destination
    (2 x `mib` MiB) stay resident in L2: the rate that bounds a kernel whose
    working set L2 serves."""
    import torch
    a = torch.empty(mib << 18, dtype=torch.float32, device=dev).fill_(1.0)
    b = torch.empty_like(a)
    for _ in range(20):
        b.copy_(a)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        b.copy_(a)
    e1.record()
    torch.cuda.synchronize(dev)
    return 2 * a.numel() * 4 * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9


DECODE_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")


def load_decode_traffic():
    """DRAM / L2 bytes per decode step from a committed ncu summary, only if
    it was taken on the current kernel source."""
    try:
        with open(DECODE_TRAFFIC_FILE) as f:
            t = json.load(f)
        if t.get("kernel_sha256_16") == kernel_hash():
            return t
    except Exception:
        pass
    return None


def decode_leg(dev, mm, flushed_steps=50):
    """Batched generation on a (128, 5120, 16) fp32 state (42 MB) with fresh
    bf16 inputs per step (16 distinct input sets cycled).

    warm: 1024 steps replayed from one CUDA graph.  The state stays resident
    in the 126 MB L2 across steps, so this figure is bound by L2, and it is
    reported against an L2-resident copy rate measured alongside.
    flushed: single steps timed one by one (CUDA events around each), with
    L2 flushed (a write of twice its size) before each, so the state comes
    from HBM; reported against the measured HBM copy rate."""
    import torch
    shp = synth.DECODE
    par = synth.decode_params(shp)
    A = torch.from_numpy(par["A"]).to(dev)
    dtb = torch.from_numpy(par["dt_bias"]).to(dev)
    dsk = torch.from_numpy(par["D_skip"]).to(dev)
    sets = []
    for i in range(16):
        si = synth.decode_step_inputs(shp, i)
        sets.append([synth.to_torch(si[k], shp.dtype, dev) for k in ("x", "delta", "z", "B", "C")])
    state = torch.zeros((shp.batch, shp.dim, shp.dstate), device=dev)
    y = torch.empty((shp.batch, shp.dim), dtype=torch.bfloat16, device=dev)
    steps = shp.steps
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for i in range(3):
            x, dl, z, Bt, Ct = sets[i % 16]
            mm.mamba_state_update(state, x, dl, dtb, A, Bt, Ct, dsk, z, y=y, stream=s)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(steps):
            x, dl, z, Bt, Ct = sets[i % 16]
            mm.mamba_state_update(state, x, dl, dtb, A, Bt, Ct, dsk, z, y=y, stream=s)
    g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 3
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    warm_us = e0.elapsed_time(e1) * 1e3 / (reps * steps)

    # flushed: the state leaves L2 before every timed step
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    cur = torch.cuda.current_stream(dev)
    times = []
    for i in range(flushed_steps + 3):
        flush.fill_(float(i))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x, dl, z, Bt, Ct = sets[i % 16]
        ev0.record(cur)
        mm.mamba_state_update(state, x, dl, dtb, A, Bt, Ct, dsk, z, y=y, stream=cur)
        ev1.record(cur)
        torch.cuda.synchronize(dev)
        if i >= 3:
            times.append(ev0.elapsed_time(ev1) * 1e3)
    flushed_us = statistics.median(times)
    del flush

    bytes_step = 2 * shp.state_bytes() + shp.io_bytes_per_step()
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    l2_gbs = l2_copy_rate(dev)
    warm_gbs = bytes_step / (warm_us * 1e-6) / 1e9
    flushed_gbs = bytes_step / (flushed_us * 1e-6) / 1e9
    out = {"workload": shp.name, "bytes_per_step": bytes_step,
           "bytes_note": "state read + write (2 x 41.9 MB) + x, delta, z, y, B, C",
           "l2_bytes": l2,
           "warm": {"us_per_step": warm_us, "tokens_per_s": shp.batch / (warm_us * 1e-6),
                    "GB/s": warm_gbs, "bound": "l2", "l2_copy_GB/s": l2_gbs,
                    "frac_of_l2_copy": warm_gbs / l2_gbs, "graph_steps": steps,
                    "note": "the 42 MB state stays resident in L2 across graph-replayed steps"},
           "flushed": {"us_per_step": flushed_us, "tokens_per_s": shp.batch / (flushed_us * 1e-6),
                       "GB/s": flushed_gbs, "bound": "hbm", "peak_GB/s": hbm,
                       "hbm_frac": flushed_gbs / hbm, "peak_source": src, "steps": flushed_steps,
                       "note": "L2 flushed before each step; single launches timed one by one, "
                               "so launch latency is included"}}
    t = load_decode_traffic()
    out["traffic"] = t if t is None else {k: t[k] for k in t if k != "kernel_sha256_16"}
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(synth.SCAN_SHAPES), default="m2p8")
    ap.add_argument("--soak", type=float, default=1.0, help="untimed seconds before warm-up")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-ext", action="store_true")
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--no-conv", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layout", type=int, choices=[0, 1, 2], default=0,
                    help="scan kernel for dstate 9..16: 0 automatic, 1 lane per channel, "
                         "2 state split over four warps")
    ap.add_argument("--decode-only", action="store_true",
                    help="only run the decode leg (warm and flushed) and print it")
    ap.add_argument("--pipe-rates", action="store_true",
                    help="only measure the per-SM arithmetic rates the roofline is built on")
    args = ap.parse_args()
    if args.pipe_rates:
        return run_pipe_rates()
    if args.decode_only:
        import torch
        torch.cuda.set_device(0)
        import selective_state_space_135_b300 as mm
        print(json.dumps({"decode": decode_leg(torch.device("cuda", 0), mm)}), flush=True)
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    shape = synth.SCAN_SHAPES[args.workload]
    if args.impl == "reference":
        return run_reference(args, shape)
    return run_ours(args, shape)


if __name__ == "__main__":
    sys.exit(main())
