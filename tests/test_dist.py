"""The multi-rank bench logic on CPU with two gloo ranks: each rank runs its
own seeded replica of the workload, the step time is the slowest rank's, and
the job value counts the units of every rank."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from exact_second_order_gb300 import inputs as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 10.0 + 5.0 * rank  # rank 1 is slower
        mx = bench.reduce_max(my_ms, world)
        w = bench.rank_workload(wl.small_workload(1, 2, 16, 8, "bf16"), rank)
        x = wl.make_inputs(w)
        out[rank] = (mx, bench.job_tflops(1e12, 4, world, mx), w.seed, float(x["Q"].float().sum()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    (mx0, v0, s0, q0), (mx1, v1, s1, q1) = out[0], out[1]
    assert mx0 == mx1 == 15.0                      # the slowest rank sets the time
    assert v0 == v1 == pytest.approx(2 * 1e12 * 4 / 15e-3 / 1e12)
    assert (s0, s1) == (0, 1) and q0 != q1         # independent units per rank


def test_single_rank_helpers():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.job_tflops(2e12, 10, 1, 1000.0) == pytest.approx(20.0)
