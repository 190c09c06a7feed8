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


def test_reference_arm_whole_workload(monkeypatch, capsys):
    """By default the oracle runs the arm's whole workload every step."""
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    args = _Args()
    args.reference_tokens = 0
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip())
    assert line["config"]["sample_tokens"] is None
    assert "whole workload" in line["cpu_baseline"]["sample"]
    assert line["value"] > 0


def test_reference_arm_packed_sample_keeps_sequences(monkeypatch, capsys):
    """A packed workload's sample keeps every sequence apart (its first
    tokens), with the offsets of the sample."""
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    args = _Args()
    args.workload = "varlen8_h12"
    args.reference_tokens = 16
    args.steps = 1
    args.warmup = 0
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip())
    assert line["config"]["sample_tokens"] == 16
    assert "first 16 tokens" in line["cpu_baseline"]["sample"]


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(_Args())
    assert capsys.readouterr().out == ""


def test_call_roofline_counts_only_algorithmic_bytes():
    """The headline fraction divides the path's algorithmic bytes (1,538 B per
    head-token plus the states) by the whole call's time; packets and
    segment states appear only as workspace bytes."""
    T, H = 8192, 6
    inp = {"N": 1, "q": torch.empty((1, T, H, 1)), "cu_seqlens": None,
           "init_state": torch.empty((1, H, 1, 1))}
    ht = T * H
    r = bench.call_roofline(inp, ht, H, 25, False, 100.0, (0.03, 0.03, 0.015, 0.025), 6673.8,
                            "measured", 1925.9, "measured", "t8192_h6", 0)
    path = 1538 * ht + 2 * H * 128 * 128 * 2
    assert r["algorithmic_bytes"] == path
    assert abs(r["achieved"] - path / 100e-6 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 6673.8) < 1e-12
    assert 0.11 < r["frac"] < 0.12
    assert abs(r["tensor"]["frac"] - 117760 * ht / 100e-6 / 1e12 / 1925.9) < 1e-12
    assert r["dominant_kernel"] == "chunk_prep"   # first of the two 30-us kernels
    assert set(r["kernels"]) == {"chunk_prep", "transition", "segment_chain", "recurrence"}
    # each kernel counts the method bytes it touches: v is read by the
    # transition pass and again by the rerun, everything else once
    assert sum(k["method_bytes"] for k in r["kernels"].values()) == path + 256 * ht
    assert r["kernels"]["recurrence"]["workspace_bytes"] >= 864 * ht
    # serial plan: preparation and recurrence split the path's bytes exactly
    r = bench.call_roofline(inp, ht, H, 0, False, 700.0, (0.3, 0.0, 0.0, 0.4), 6673.8,
                            "measured", 1925.9, "measured", "t8192_h6", 0)
    assert sum(k["method_bytes"] for k in r["kernels"].values()) == path
    assert r["dominant_kernel"] == "recurrence"


def test_profiled_traffic_entries_match_sources():
    """Every measured-traffic entry still matches the sources it was captured
    from (a changed kernel needs a new capture or loses its entry), and the
    figures are reported for the default engine only."""
    for (kernel, workload), (nbytes, files, _digest) in bench.PROFILED_TRAFFIC.items():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, "kimi_delta_attention_kda_gb300", "csrc", f)), f
        assert bench.profiled_traffic(kernel, workload, 0) == nbytes, (kernel, workload)
        assert bench.profiled_traffic(kernel, workload, 2) is None
    assert bench.profiled_traffic("chunk_prep", "no_such_workload", 0) is None
