"""The benchmark's multi-GPU path is independent replicas: a barrier around the timed
region and the max of the ranks' times are its only cross-rank operations.  Checked here
with two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.DistCtx()
    d.init("gloo")
    d.barrier()
    got = d.max(1.5 + rank)          # each rank's "seconds"
    out[rank] = got
    d.barrier()
    d.done()


def test_two_gloo_ranks_take_the_max_time():
    import torch.multiprocessing as mp
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    d = bench.DistCtx()
    args = type("A", (), {"workload": "taylor_green_32", "steps": 1, "warmup": 3})()
    assert bench.run_reference(args, d) is None
