"""Multi-rank host logic of bench.py on CPU with two gloo ranks.

The benchmark runs independent replicas under torchrun: it takes the slowest
rank's time and reports all ranks' units over it.  These tests run that logic
with the gloo backend on CPU (no GPU, no NCCL).
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        ms_rank = 10.0 + 5.0 * rank              # rank 1 is the slower one
        value, ms = bench.job_throughput(world, 8192, ms_rank)
        bench.barrier(world)
        out[rank] = (value, ms)
    finally:
        dist.destroy_process_group()


def test_two_rank_throughput_uses_slowest_rank():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in (0, 1):
        value, ms = res[rank]
        assert ms == pytest.approx(15.0)
        assert value == pytest.approx(2 * 8192 / 15e-3)


def test_single_rank_throughput():
    import bench
    value, ms = bench.job_throughput(1, 1000, 2.0)
    assert ms == 2.0 and value == pytest.approx(500_000.0)


def test_reference_arm_prints_only_on_rank_zero(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 3
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
