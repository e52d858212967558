"""The multi-process side of bench.py on CPU (gloo, world size 2): the job time is the
slowest rank's, and the reference arm runs on rank 0 only. Replicas only: no data-path
collective exists to test."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    got = bench.max_over_ranks(1.5 + rank, w)
    dist.barrier()
    out[rank] = (r, w, local, got)
    dist.destroy_process_group()


def test_job_time_is_the_slowest_rank():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == (0, 2, 0, 2.5)
    assert out[1] == (1, 2, 1, 2.5)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """A rank other than 0 leaves the reference arm at once, before touching the oracle."""
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    import argparse
    args = argparse.Namespace(impl="reference", workload="tiny", rows=None, steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args) is None
