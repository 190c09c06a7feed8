"""Host logic of bench.py that needs no GPU: the reference arm (the oracle)
and the multi-rank bookkeeping, with two gloo processes on the CPU: every
rank gets the slowest rank's time, the job rate counts every rank's units,
and under torchrun only rank 0 runs and prints the reference arm."""

import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        # rank r "measured" 10 + r ms of kernels and 30 - r ms end to end
        got = bench.max_over_ranks([10.0 + rank, 30.0 - rank], torch.device("cpu"))
        out[rank] = got + [bench.job_throughput(world, 1000, 5, got[0])]
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_processes():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    for rank in (0, 1):
        t_kernel, t_e2e, rate = res[rank]
        assert t_kernel == 11.0 and t_e2e == 30.0
        assert rate == pytest.approx(2 * 1000 * 5 / 11e-3)


def test_single_process_is_identity():
    assert bench.max_over_ranks([3.0, 4.5], torch.device("cpu")) == [3.0, 4.5]
    assert bench.job_throughput(1, 100, 2, 4.0) == pytest.approx(100 * 2 / 4e-3)


class _Args:
    workload = "t256_h1"
    steps = 2
    warmup = 1
    reference_tokens = 64


def test_reference_arm_rank0_line(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    bench.run_reference(_Args())
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == "head-tokens/s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["config"]["sample_tokens"] == 64


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(_Args())
    assert capsys.readouterr().out == ""
