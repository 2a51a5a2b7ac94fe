"""The bench's multi-rank host logic on CPU with two gloo ranks: the job's time
is the slowest rank's, its throughput counts every rank's work, and only rank
0 of the reference arm does any work."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.slowest_rank_ms(1.0 + rank, world, "cpu")      # rank r took 1 + r ms
        out[rank] = (ms, bench.job_tflops(world, 1e12, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_value():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        got = dict(out)
    assert got[0] == got[1] == (2.0, pytest.approx(1000.0))   # 2 ranks x 1 TFLOP over 2 ms


def test_reference_arm_rank_other_than_zero_does_no_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "cpu_sample_time", lambda *a, **k: called.append(1))
    args = type("A", (), {"steps": 2, "warmup": 1, "gpus": 2})()
    assert bench.run_reference(args) == 0 and not called
