"""The benchmark's multi-process path on CPU: two gloo ranks on 127.0.0.1.

The hot path shards by request with no exchange, so N GPUs run N replicas of
the workload (weak scaling).  What crosses ranks is the timing: the job's
step time is the slowest rank's, and the whole-job value counts every rank's
bytes.  These tests run that logic as real processes with the gloo backend.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_loc_gb300 import workloads as W


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        local_ms = 1.0 + 0.5 * rank   # rank 1 is the slow one
        job_ms = bench.job_step_ms(torch, local_ms, "cpu")
        case = W.tiny_decode()
        per_rank = bench.decode_bytes(case)
        out[rank] = (job_ms, bench.job_value_gbs(world, per_rank, job_ms), per_rank)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_and_value_counts_every_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 1.5             # max over ranks, seen by every rank
    per_rank = res[0][2]
    assert res[0][1] == res[1][1] == world * per_rank / 1.5e-3 / 1e9


def test_single_process_job_time_is_local():
    assert not dist.is_initialized()
    assert bench.job_step_ms(torch, 2.25, "cpu") == 2.25
    assert bench.job_value_gbs(1, 1e9, 1.0) == 1000.0


def test_rank_workloads_have_equal_shapes_and_different_values():
    """Weak scaling: each rank decodes its own copy of the batched workload."""
    a = W.batched_decode(batch=4, lo=16, hi=64, size=1024, seed=bench.rank_seed(0))
    b = W.batched_decode(batch=4, lo=16, hi=64, size=1024, seed=bench.rank_seed(1))
    assert bench.rank_seed(0) != bench.rank_seed(1)
    assert a.q.shape == b.q.shape and a.k_buffer.shape == b.k_buffer.shape
    assert not np.array_equal(a.q, b.q)


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    """Under a launcher, ranks other than 0 leave the reference arm at once."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.run_reference(None) is None
    assert capsys.readouterr().out == ""
