"""The benchmark's multi-rank host logic on CPU: two gloo ranks.

Requests are independent, so the path shards by request with no data-path
collective: every rank drafts and verifies its own block of request ids, and
the job's time is the slowest rank's (a max over ranks).  These tests run
that logic with world_size 2 on the gloo backend, rendezvous on 127.0.0.1.
"""
import os
import socket
import sys
import types

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, R, gamma, steps):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ids = bench.rank_request_ids(R, rank)
        assert ids.dtype == np.uint32 and ids.shape == (R,)
        # every rank's ids, gathered: disjoint blocks covering 0 .. world R - 1
        t = torch.from_numpy(ids.astype(np.int64))
        got = [torch.empty_like(t) for _ in range(world)]
        dist.all_gather(got, t)
        allids = torch.cat(got).numpy()
        assert np.array_equal(np.sort(allids), np.arange(world * R))
        # the slowest rank's time is the job's
        local_ms = 10.0 + 7.5 * rank
        m = bench.max_over_ranks(local_ms, world)
        assert m == 10.0 + 7.5 * (world - 1)
        v = bench.job_throughput(R * gamma, world, steps, m)
        assert abs(v - R * gamma * world * steps / (m / 1000.0)) <= 1e-9 * v
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_requests_and_take_the_slowest():
    mp.start_processes(_worker, args=(2, _free_port(), 256, 5, 4), nprocs=2, join=True, start_method="spawn")


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert np.array_equal(bench.rank_request_ids(4, 0), np.arange(4, dtype=np.uint32))
    assert bench.job_throughput(1280, 1, 20, 1000.0) == 1280 * 20


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun only rank 0 runs the oracle arm; the others exit 0 at once."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = types.SimpleNamespace(workload="headline", steps=1, warmup=3)
    assert bench.run_reference(args) == 0


def test_gpu_arm_refuses_several_ranks(monkeypatch, capsys):
    """The GPU arm runs on one GPU only (its kernels share W2 tiles within a
    cluster by multicast over this GPU's memory): under torchrun with two ranks
    rank 0 prints one line saying so and every rank exits 0 without work."""
    import json
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "0")
    assert bench.main(["--gpus", "2"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["n_gpus"] == 2 and line["value"] is None and "one GPU" in line["unavailable"]
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--gpus", "2"]) == 0
    assert capsys.readouterr().out.strip() == ""
