"""The multi-GPU bench path on the CPU: two gloo ranks, host logic only.

Each rank of a multi-GPU run holds an independent replica of the workload (the jagged
batch has no exchange between sequences), so the only cross-rank steps are the timing
reduction (the job is as slow as its slowest replica) and the whole-job throughput.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.5 + rank, world, "cpu")
        dist.barrier()
        value = bench.job_tflops(2.0e12, world, slowest * 1e-3)
        out.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_job_value():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    # both ranks see the slower replica's time, and the value counts both replicas' work
    assert [r[1] for r in res] == [2.5, 2.5]
    for _, slowest, value in res:
        assert value == pytest.approx(2 * 2.0e12 / (slowest * 1e-3) / 1e12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_tflops(1e12, 1, 1e-3) == pytest.approx(1000.0)


def test_replicas_share_shapes_not_values():
    w = workloads.WORKLOADS["tiny"]
    lq, lk = workloads.lengths(w.name, seed=0)
    b0 = workloads.make_batch(w, lq, lk, seed=bench.replica_seed(0))
    b1 = workloads.make_batch(w, lq, lk, seed=bench.replica_seed(1))
    assert np.array_equal(b0["offs_q"], b1["offs_q"])
    for k in ("q", "k", "v", "do"):
        assert b0[k].shape == b1[k].shape
        assert not torch.equal(b0[k], b1[k])
