"""The multi-rank bookkeeping of bench.py, run as two gloo ranks on the CPU:
each rank scans its own independently seeded batch (weak scaling, no
data-path collective), the timed region is the slowest rank's, and the
whole-job rate counts the elements of every rank."""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shape = synth.M2P8
        ms_local = 10.0 + 5.0 * rank                       # rank 1 is the slow one
        ms = bench.max_over_ranks(ms_local, dist, "cpu")
        rate = bench.whole_job_rate(shape.elems, 7, world, ms)
        # each rank's inputs: a small seeded slice of its own copy of the workload
        seed = bench.rank_seed(shape, rank)
        u0 = synth.normal(seed, "u", (4,))
        dist.barrier()
        out[rank] = (ms, rate, seed, u0.tolist())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    (ms0, rate0, seed0, u0), (ms1, rate1, seed1, u1) = res[0], res[1]
    assert ms0 == ms1 == 15.0                       # max over ranks
    assert rate0 == rate1 == pytest.approx(synth.M2P8.elems * 7 * 2 / 15e-3)
    assert seed0 != seed1 and not np.allclose(u0, u1)   # independent replicas


def test_single_rank_is_local():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(100, 2, 1, 1.0) == pytest.approx(2e5)
