"""Benchmark of GB300-native KDA prefill (head-tokens/s and us per call).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one kda_prefill call (all of its kernels) over one batch of
synthetic input already resident in HBM; by default the timed steps replay
the call captured once in a CUDA graph (`--graph 0`: eager calls; the eager
time is reported beside it either way).  The default workload is B=1, H=6,
T=8192, d=128 ("FlashKDA column split", section 4: the small-head
tensor-parallel shard at 8,192 tokens); a secondary line item times B=1,
H=96, T=8192 the same way.  Between timed steps a 512 MiB buffer is written
to flush the 129 MB L2.

Reported: `value` = head-tokens/s over the timed steps (device time, CUDA
events on the launching stream); `e2e` = the same metric through the host-buffer
entry point kda_prefill_host (pinned host tensors; the library copies the
inputs in and O and the final state out inside every timed step, overlapped
with the computation); `roofline`: the whole call against its algorithmic
bytes (1,538 B per head-token plus the states) at the measured copy
bandwidth, the tensor fraction of its algorithmic FLOPs, per-kernel times
(events recorded by the library between its kernels in a separate pass of
eager calls) with each kernel's method and workspace bytes, and
`roofline.critical_path` (HBM, tensor and serial-chain bounds of the call); `cpu_baseline` = the FP64 oracle timed on this host's cores.  `--impl reference` times that oracle
alone on a bounded sample of the same workload (the pages name no runnable
reference implementation).  Under torchrun every rank runs its own replica of
the workload on its own GPU (weak scaling, no collective in the data path).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from kimi_delta_attention_kda_gb300 import synthetic  # noqa: E402

METRIC = "KDA prefill head-tokens/sec and us/call at T=8192, H=6 and H=96 (GB300)"
UNIT = "head-tokens/s"
# Page numbers for this workload (B200, both kernels, T=8192; "FlashKDA column
# split", section 4): FlashKDA 731.7 us at H=6 and 1,032.6 us at H=96.
FLASHKDA_B200_US = {"t8192_h6": 731.7, "t8192_h96": 1032.6}
COLUMN_SPLIT_B200_US = {"t8192_h6": 283.4, "t8192_h96": 914.7}
L2_FLUSH_BYTES = 512 << 20

# Algorithmic bytes per head-token of the path (the method's own inputs and
# outputs, nothing the implementation adds): q, k, v 256 B each, g 512 B,
# beta 2 B, O 256 B; plus 32 KB per (sequence, head) per state read or
# written.  The 13,824-byte packet per 16 tokens (864 B per head-token) that
# the preparation writes and the recurrence reads is workspace.
PACKET_PER_TOKEN = 13824 / 16
PATH_BYTES_PER_HT = 2 * 256 + 512 + 2 + 256 + 256
STATE_BYTES = 128 * 128 * 2

# DRAM bytes (read + write) of one launch of each kernel (of the segment
# chain: its launches in one call; of the packed recurrence: both concurrent
# launches), from one ncu capture each (summaries in profiles/).  A figure is
# reported only while the kernel's sources still hash to the value they had
# when it was captured (or, where a file changed elsewhere, re-keyed once the
# kernel's own code was checked unchanged: the quad recurrence beside the
# transition pass in kda_recurrence.cu).
REC_SOURCES = ("kda_recurrence.cu", "kda_rec_impl.cuh", "kda_common.cuh", "kda_segmap.cuh")
PREP_SOURCES = ("kda_prep.cu", "kda_prep_impl.cuh", "kda_common.cuh")
SEG_SOURCES = ("kda_segments.cu", "kda_common.cuh", "kda_segmap.cuh")
FUSED_SOURCES = ("kda_fused.cu", "kda_prep_impl.cuh", "kda_rec_impl.cuh", "kda_common.cuh")
PROFILED_TRAFFIC = {
    ("chunk_prep", "t8192_h6"): (52.8e6, PREP_SOURCES, "49c80c6456fccd98"),
    ("transition", "t8192_h6"): (55.4e6, REC_SOURCES, "76dc6fcc5db481ea"),
    ("segment_chain", "t8192_h6"): (10.0e6, SEG_SOURCES, "14ee7f8b9ec3c9c7"),
    ("recurrence", "t8192_h6"): (61.0e6, REC_SOURCES, "76dc6fcc5db481ea"),
    ("fused", "t8192_h96"): (1854.1e6, FUSED_SOURCES, "e007fafac3c3037e"),
    ("chunk_prep", "t8192_h96"): (1454.6e6, PREP_SOURCES, "49c80c6456fccd98"),
    ("recurrence", "t8192_h96"): (1067.0e6, REC_SOURCES, "76dc6fcc5db481ea"),
    ("fused", "t256_h1"): (0.4e6, FUSED_SOURCES, "e007fafac3c3037e"),
    ("fused", "varlen8_h12"): (681.3e6, FUSED_SOURCES, "e007fafac3c3037e"),
}


def profiled_traffic(kernel, workload, engine):
    import hashlib
    entry = PROFILED_TRAFFIC.get((kernel, workload))
    if entry is None or engine != 0:   # the figures are for the default kernels
        return None
    nbytes, files, digest = entry
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "kimi_delta_attention_kda_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return nbytes if h.hexdigest()[:16] == digest else None


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def device_inputs(inp, device):
    return {k: (None if inp[k] is None else inp[k].to(device))
            for k in ("q", "k", "v", "g", "beta", "init_state", "cu_seqlens")}


def head_tokens(inp):
    return int(inp["q"].shape[0] * inp["q"].shape[1] * inp["q"].shape[2])


def time_kernel_steps(kda, d, steps, warmup, flush, stream, profile=False, graph=False):
    """Device time of `steps` kda_prefill calls (L2 flushed before each).
    With `graph`, the call is captured once into a CUDA graph after the
    warm-up and every step replays it (the flush stays outside the graph)."""
    out = torch.empty_like(d["v"])
    N = d["init_state"].shape[0] if d["init_state"] is not None else d["q"].shape[0]
    if d["cu_seqlens"] is not None:
        N = d["cu_seqlens"].numel() - 1
    H = d["q"].shape[2]
    fin = torch.empty((N, H, 128, 128), dtype=torch.bfloat16, device=d["q"].device)

    def eager():
        kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                        cu_seqlens=d["cu_seqlens"], out=out, final_state=fin, stream=stream)

    call = eager
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.zero_()
            eager()
        stream.synchronize()
        launches = kda._lib.last_call_launches()   # kernels one call enqueues
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                eager()
            stream.synchronize()
            call = g.replay
            # Untimed replays: the first launches of a new graph upload it.
            for _ in range(min(warmup, 3)):
                flush.zero_()
                call()
            stream.synchronize()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        if profile:
            kda._lib.profile_begin(steps)
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            call()
            ends[i].record(stream)
        stream.synchronize()
        prof = kda._lib.profile_end_detail() if profile else None
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return ms, prof, launches


def time_e2e_steps(kda, inp, steps, warmup, flush, stream, device):
    """Same metric through the public API with host buffers: every step is one
    kda_prefill_host call on pinned host tensors, which copies the inputs to
    the device, computes, and copies O and the final state back (the library
    overlaps those copies with the computation)."""
    host = {k: (None if inp[k] is None else inp[k].pin_memory())
            for k in ("q", "k", "v", "g", "beta", "init_state", "cu_seqlens")}
    H = inp["q"].shape[2]
    N = inp["N"]
    out_h = torch.empty(host["v"].shape, dtype=torch.bfloat16).pin_memory()
    fin_h = torch.empty((N, H, 128, 128), dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = out_h.numel() * 2 + fin_h.numel() * 2

    def step():
        kda.kda_prefill_host(host["q"], host["k"], host["v"], host["g"], host["beta"],
                             host["init_state"], cu_seqlens=host["cu_seqlens"], out=out_h,
                             final_state=fin_h, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.zero_()
            step()
        stream.synchronize()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        stream.synchronize()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return ms, h2d, d2h


def cpu_baseline(name, min_seconds=10.0):
    """The FP64 oracle, as it stands, on this host's cores, over the whole
    workload repeated until about `min_seconds` of CPU work have run."""
    import oracle
    inp = synthetic.make_workload(name)
    cu = inp["cu_seqlens"]
    reps, total = 0, 0.0
    while total < min_seconds and reps < 100:
        t0 = time.perf_counter()
        oracle.kda_token(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["init_state"],
                         cu_seqlens=None if cu is None else cu.numpy())
        total += time.perf_counter() - t0
        reps += 1
    ht = head_tokens(inp)
    return {"value": ht * reps / total, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "the whole %s workload (%d head-tokens) run %d times, FP64 token recurrence"
                      % (inp["workload"].name, ht, reps)}


def run_reference(args):
    """The oracle as the reference arm, on this arm's workload: every step the
    whole workload (the default, reference_tokens 0), or with reference_tokens
    > 0 the first that many tokens of every sequence (a quicker sample)."""
    import oracle
    ws, rank, _ = dist_env()
    if ws > 1 and rank != 0:
        return
    inp = synthetic.make_workload(args.workload)
    H = inp["q"].shape[2]
    init = inp["init_state"]
    if args.reference_tokens <= 0:
        sl = {k: inp[k] for k in ("q", "k", "v", "g", "beta")}
        cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].numpy()
        ht = head_tokens(inp)
        sample = "the whole workload %s every step (%d head-tokens), FP64 token recurrence" % (
            inp["workload"].name, ht)
        tokens = inp["q"].shape[1]
    else:
        # The first `tokens` of every sequence (packed: of each sequence's span).
        tokens = min(inp["q"].shape[1], args.reference_tokens)
        if inp["cu_seqlens"] is None:
            sl = {k: inp[k][:, :tokens].contiguous() for k in ("q", "k", "v", "g", "beta")}
            cu = None
        else:
            c = inp["cu_seqlens"].tolist()
            spans = [(c[n], min(c[n + 1], c[n] + tokens)) for n in range(len(c) - 1)]
            sl = {k: torch.cat([inp[k][:, a:b] for a, b in spans], 1).contiguous()
                  for k in ("q", "k", "v", "g", "beta")}
            lens = [b - a for a, b in spans]
            cu = [0]
            for n in lens:
                cu.append(cu[-1] + n)
            import numpy as np
            cu = np.asarray(cu, dtype=np.int64)
        ht = int(sl["q"].shape[0] * sl["q"].shape[1] * H)
        sample = ("first %d tokens of every sequence of %s (%d head-tokens per step), FP64 token "
                  "recurrence" % (tokens, inp["workload"].name, ht))

    def step():
        oracle.kda_token(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], init, cu_seqlens=cu)

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = ht * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": inp["workload"].name,
                   "sample_tokens": None if args.reference_tokens <= 0 else tokens},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(values, device):
    """Each value's maximum over the ranks of the default process group (the
    values themselves with one process): the slowest replica sets the time."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(world_size, units_per_rank, steps, total_ms):
    """Whole-job rate: every rank's units over the slowest rank's time."""
    return world_size * units_per_rank * steps / (total_ms * 1e-3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense BF16 TFLOP/s (burst) from MEASURED_PEAKS.json, else the recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


# Algorithmic FLOPs per head-token of the chunkwise form at C = 16 (dense
# 16-tiles): the three 128 x 128 x 16 state products per chunk, the A^qk and R
# scores, U (A^kk)^T and U (A^qk)^T, and the 16 x 16 inverse, per 16 tokens.
FLOP_PER_HT = (3 * 2 * 128 * 128 * 16 + 2 * 65536 + 2 * 65536 + 49152) / 16


def critical_path(kda, inp, ht, state_io, us_per_call, segs):
    """Bounds on the call: HBM (the path's algorithmic bytes at the measured
    copy bandwidth), tensor (its FLOPs at the measured BF16 rate) and the
    serial chain (the longest sequence's chunk steps times the measured
    shortest dependent chunk-step chain); `frac` = the largest over the time.
    A segmented call is not a serial walk: its own chain bound is the two
    walks of one segment's L chunks (`plan_*`), which the serial bound can
    exceed."""
    t_step = kda._lib.chain_step_ns()
    if inp["cu_seqlens"] is None:
        steps = int(math.ceil(inp["q"].shape[1] / 16))
    else:
        cu = inp["cu_seqlens"].tolist()
        steps = max((cu[i + 1] - cu[i] + 15) // 16 for i in range(len(cu) - 1))
    hbm_gbs, _ = measured_peaks()
    tflops, tkind = measured_tensor_peak()
    hbm_us = (PATH_BYTES_PER_HT * ht + state_io) / (hbm_gbs * 1e3)
    tensor_us = FLOP_PER_HT * ht / (tflops * 1e6)
    chain_us = steps * t_step / 1e3
    bound = max(hbm_us, tensor_us, chain_us)
    kind = "chain" if bound == chain_us else ("hbm" if bound == hbm_us else "tensor")
    res = {"t_step_ns": t_step, "chain_steps": steps, "chain_bound_us": chain_us,
           "hbm_bound_us": hbm_us, "tensor_bound_us": tensor_us, "tensor_peak_kind": tkind,
           "bound_us": bound, "bound": kind, "frac": bound / us_per_call,
           "plan": "segmented" if segs else "serial"}
    if segs:
        if inp["cu_seqlens"] is None:
            L = int(math.ceil(steps / segs))
        else:   # the planner's segment length from its bound on all segments
            n = inp["cu_seqlens"].numel() - 1
            c_ub = (inp["q"].shape[1] + 15 * n) // 16
            L = int(math.ceil(c_ub / max(segs - n, 1)))
        plan_chain = 2 * L * t_step / 1e3
        plan_bound = max(hbm_us, tensor_us, plan_chain)
        res.update({"plan_segment_chunks": L, "plan_chain_bound_us": plan_chain,
                    "plan_bound_us": plan_bound, "plan_frac": plan_bound / us_per_call,
                    "note": "bound/frac: a serial walk's bounds, which a segmented call is not "
                            "held to (frac > 1 when it beats the serial chain); plan_*: the "
                            "bounds of the segmented plan that ran"})
    return res


def call_roofline(inp, ht, H, segs, fused, us_call, prof_ms, peak, peak_kind, tpeak,
                  tpeak_kind, workload, engine):
    """Roofline of one call against the path's algorithmic bytes and FLOPs.

    Algorithmic bytes are the method's own inputs and outputs: q, k, v (256 B
    per head-token each), g (512 B), beta (2 B) and O (256 B), 1,538 B per
    head-token, plus 32 KB per (sequence, head) for each state read or
    written.  The packets that pass from the preparation to the recurrence,
    and the segmented scan's intermediate states, are workspace: they are
    counted separately and never in `achieved`.  `frac` = achieved / the
    measured copy bandwidth over the whole call; per kernel, `method_frac`
    counts only the method bytes that kernel reads or writes.  `traffic` is
    the DRAM bytes ncu measured for every kernel of one call (null unless all
    of the call's kernels have a current capture)."""
    prep_ms, trans_ms, chain_ms, rec_ms = prof_ms
    n_states = inp["N"] * H
    state_io = (2 if inp["init_state"] is not None else 1) * n_states * STATE_BYTES
    seg_states = n_states * segs * STATE_BYTES
    path_bytes = PATH_BYTES_PER_HT * ht + state_io
    flops = FLOP_PER_HT * ht
    pkt = PACKET_PER_TOKEN * ht
    in_qkgb = (2 * 256 + 512 + 2) * ht
    vo = 2 * 256 * ht
    # name: (mean ms, method bytes, workspace bytes)
    if fused:
        kernels = {"fused": (rec_ms, path_bytes, 0.0)}
    elif segs:
        kernels = {"chunk_prep": (prep_ms, in_qkgb, pkt),
                   "transition": (trans_ms, 256 * ht, pkt + 2 * seg_states),
                   "segment_chain": (chain_ms, state_io, 3 * seg_states),
                   "recurrence": (rec_ms, vo, pkt + seg_states)}
    else:
        kernels = {"chunk_prep": (prep_ms, in_qkgb, pkt),
                   "recurrence": (rec_ms, vo + state_io, pkt)}
    total_ms = sum(k[0] for k in kernels.values())
    per = {}
    traffic = 0.0
    for name, (ms, mb, wb) in kernels.items():
        tr = profiled_traffic(name, workload, engine)
        per[name] = {"us": 1e3 * ms, "share": ms / total_ms if total_ms > 0 else None,
                     "method_bytes": mb, "workspace_bytes": wb,
                     "method_frac": mb / (ms * 1e-3) / 1e9 / peak if ms > 0 else None,
                     "traffic": tr}
        traffic = None if (traffic is None or tr is None) else traffic + tr
    dom = max(kernels, key=lambda k: kernels[k][0])
    achieved = path_bytes / (us_call * 1e-6) / 1e9
    tflops = flops / (us_call * 1e-6) / 1e12
    return {
        "bound": "hbm", "scope": "whole call (every kernel of one kda_prefill)",
        "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
        "peak_kind": peak_kind, "algorithmic_bytes": path_bytes,
        "algorithmic_state_bytes": state_io,
        "traffic": traffic,
        "workspace_traffic": None if traffic is None else traffic - path_bytes,
        "tensor": {"flops": flops, "achieved_tflops": tflops, "peak_tflops": tpeak,
                   "frac": tflops / tpeak, "peak_kind": tpeak_kind},
        "dominant_kernel": dom,
        "dominant_kernel_path_frac": path_bytes / (kernels[dom][0] * 1e-3) / 1e9 / peak,
        "kernels": per,
        "chain_steps": int(math.ceil(inp["q"].shape[1] / 16)) if inp["cu_seqlens"] is None
        else None,
    }


def run_ours(args):
    import kimi_delta_attention_kda_gb300 as kda
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    kda._lib.load()   # fails loudly when the library is not built
    if args.split:
        kda.set_split(args.split)
    if args.engine:
        kda.set_engine(args.engine)
    kda.set_fusion(bool(args.fusion))
    kda.set_segments(bool(args.segments))
    stream = torch.cuda.Stream(device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    inp = synthetic.make_workload(args.workload)
    d = device_inputs(inp, device)
    ht = head_tokens(inp)
    nsplit = kda.auto_split(inp["N"], inp["q"].shape[2])
    packed = inp["cu_seqlens"] is not None
    fused = kda.plan_fused(inp["N"] if packed else inp["q"].shape[0], inp["q"].shape[1],
                           inp["q"].shape[2], packed)
    segs = kda.plan_segments(inp["N"] if packed else inp["q"].shape[0], inp["q"].shape[1],
                             inp["q"].shape[2], packed)
    long_split = kda.plan_long_split(inp["N"], inp["q"].shape[1], inp["q"].shape[2]) if packed else 0

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    cvd = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    gpu_index = cvd[device.index] if device.index < len(cvd) else str(device.index)
    prof_steps = max(10, args.steps // 4)
    with ClockSampler(gpu_index) as clk:
        # The headline steps replay the call captured in a CUDA graph (with
        # --graph 1) and run without the library's profile events (an event
        # between each pair of kernels adds a few microseconds per call); a
        # second, shorter pass of eager calls records them for the per-kernel
        # split, and a third times eager calls without them.
        ms, _, launches_per_call = time_kernel_steps(kda, d, args.steps, args.warmup, flush,
                                                     stream, graph=bool(args.graph))
        _, prof, _ = time_kernel_steps(kda, d, prof_steps, 3, flush, stream, profile=True)
        eager_ms, _, _ = time_kernel_steps(kda, d, prof_steps, 3, flush, stream)
        e2e_ms, h2d, d2h = time_e2e_steps(kda, inp, args.steps, min(args.warmup, 3), flush, stream,
                                          device)
    torch.cuda.synchronize(device)
    if ws > 1:
        torch.distributed.barrier()
    status = kda.device_status(stream.cuda_stream)
    if status != 0:
        raise RuntimeError("device status %d during the benchmark" % status)

    total_ms, total_e2e = max_over_ranks([sum(ms), sum(e2e_ms)], device)
    value = job_throughput(ws, ht, args.steps, total_ms)
    e2e_value = job_throughput(ws, ht, args.steps, total_e2e)

    intervals, calls = prof
    prep_avg, trans_avg, chain_avg, rec_avg = (t / calls for t in intervals)
    peak, peak_kind = measured_peaks()
    tpeak, tpeak_kind = measured_tensor_peak()
    H = inp["q"].shape[2]
    us_call = 1e3 * total_ms / args.steps
    roofline = call_roofline(inp, ht, H, segs, fused, us_call,
                             (prep_avg, trans_avg, chain_avg, rec_avg), peak, peak_kind,
                             tpeak, tpeak_kind, args.workload, args.engine)
    state_io = roofline["algorithmic_state_bytes"]
    roofline["critical_path"] = critical_path(kda, inp, ht, state_io, us_call, segs)
    if "plan_frac" in roofline["critical_path"]:
        roofline["plan_frac"] = roofline["critical_path"]["plan_frac"]

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "us_per_call": 1e3 * total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": inp["workload"].name, "l2": "flushed (512 MiB write) before every step",
                   "recurrence_split": 1 if segs else nsplit, "recurrence_engine": args.engine,
                   "one_launch": fused, "long_sequences_at_split_2": long_split,
                   "segments_per_sequence": segs, "head_tokens_per_step": ht,
                   "kernel_times": "per-kernel split from a separate pass of %d steps with library "
                                   "events between the kernels" % prof_steps,
                   "cuda_graph": bool(args.graph)},
        "eager_us_per_call": 1e3 * sum(eager_ms) / len(eager_ms),
        "gpu_launches": launches_per_call * args.steps,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_call": 1e3 * total_e2e / args.steps,
                # The host link is shared with the machine's other work: a step now
                # and then takes tens of ms, which the mean above keeps.
                "us_per_call_median": 1e3 * sorted(e2e_ms)[len(e2e_ms) // 2],
                "entry": "kda_prefill_host"},
        "roofline": roofline,
        "clocks": clk.summary(),
    }
    if args.workload in FLASHKDA_B200_US:
        # Another machine's number: context only, never the target (vs_baseline stays null).
        line["context_b200"] = {
            "what": "FlashKDA prep + recurrence on a B200, %.1f us (pages, FlashKDA column split "
                    "section 4); not measured here" % FLASHKDA_B200_US[args.workload],
            "column_split_b200_us": COLUMN_SPLIT_B200_US[args.workload]}
    if not args.no_secondary and args.workload != "t8192_h96":
        sec = synthetic.make_workload("t8192_h96")
        ds = device_inputs(sec, device)
        ms2, _, _ = time_kernel_steps(kda, ds, max(20, args.steps // 10), 5, flush, stream,
                                   graph=bool(args.graph))
        _, prof2, _ = time_kernel_steps(kda, ds, 10, 3, flush, stream, profile=True)
        ht2 = head_tokens(sec)
        t2 = sum(ms2) / len(ms2)
        one2 = kda.plan_fused(1, sec["q"].shape[1], 96, False)
        line["secondary"] = {"workload": sec["workload"].name, "us_per_call": 1e3 * t2,
                             "value": ht2 / (t2 * 1e-3), "unit": UNIT, "one_launch": one2,
                             "recurrence_split": kda.auto_split(1, 96)}
        if one2:   # the first interval is the reset of the ready flags
            line["secondary"].update({"flag_reset_us": 1e3 * prof2[0][0] / prof2[1],
                                      "fused_us": 1e3 * sum(prof2[0][1:]) / prof2[1]})
        else:
            line["secondary"].update({"prep_us": 1e3 * prof2[0][0] / prof2[1],
                                      "recurrence_us": 1e3 * sum(prof2[0][1:]) / prof2[1]})
        sec_state = sec["N"] * 96 * STATE_BYTES * (2 if sec["init_state"] is not None else 1)
        sec_path = PATH_BYTES_PER_HT * ht2 + sec_state
        peak2, _ = measured_peaks()
        line["secondary"]["roofline"] = {
            "bound": "hbm", "scope": "whole call", "algorithmic_bytes": sec_path,
            "achieved": sec_path / (t2 * 1e-3) / 1e9, "peak": peak2, "unit": "GB/s",
            "frac": sec_path / (t2 * 1e-3) / 1e9 / peak2,
            "tensor_frac": FLOP_PER_HT * ht2 / (t2 * 1e-3) / 1e12 / measured_tensor_peak()[0]}
        del ds
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="t8192_h6", choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-tokens", type=int, default=0,
                    help="reference arm: 0 (default) runs the whole workload every step; "
                         "n > 0 the first n tokens of every sequence")
    ap.add_argument("--split", type=int, default=0,
                    help="CTAs per (sequence, head) in the recurrence (0 = automatic)")
    ap.add_argument("--engine", type=int, default=0,
                    help="recurrence engine: 0 automatic, 1 column-split warp MMA, 2 tcgen05")
    ap.add_argument("--fusion", type=int, default=1, choices=[0, 1],
                    help="allow preparation and recurrence as one launch (kda_set_fusion)")
    ap.add_argument("--graph", type=int, default=1, choices=[0, 1],
                    help="time replays of the call captured in a CUDA graph (eager calls with 0)")
    ap.add_argument("--segments", type=int, default=1, choices=[0, 1],
                    help="allow the segmented scan over chunks (kda_set_segments)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
