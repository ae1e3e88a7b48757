"""Host logic of bench.py's multi-GPU path on CPU: world size 2 over gloo.

Every rank times its own frames (weak scaling); the job's time is the
slowest rank's and its throughput counts every rank's frames.  The ranks
here report different local times so the max over ranks is observable.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 100.0 + 50.0 * rank          # rank 1 is the slowest
    total_ms, value = bench.whole_job(local_ms, frames_per_step=32, steps=10, world=world, device="cpu")
    results[rank] = (total_ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_whole_job_takes_the_slowest_rank_and_all_frames():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank, args=(world, _free_port(), results), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(results)
    assert set(res) == {0, 1}
    for total_ms, value in res.values():
        assert total_ms == pytest.approx(150.0)
        assert value == pytest.approx(2 * 32 * 10 / 0.150)


def test_whole_job_single_rank_has_no_collective():
    import bench
    total_ms, value = bench.whole_job(200.0, frames_per_step=1, steps=20, world=1)
    assert total_ms == 200.0 and value == pytest.approx(100.0)
