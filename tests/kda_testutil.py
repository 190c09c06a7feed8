"""Helpers shared by the tests: tolerance metrics, packet decoding, and oracle
runs on a subset of heads.

The tolerance for BF16 inputs and outputs with FP32 accumulation:
per (sequence, head), relative Frobenius error <= 1e-2 and max-abs error
<= 3e-2, for the output O (T_n x 128) and the final state (128 x 128); when
the reference is all zeros only the max-abs bound applies.
"""

import numpy as np
import torch

import oracle

REL_FRO_TOL = 1e-2
MAX_ABS_TOL = 3e-2

# Packet layout (bytes) of the preparation stage; see the library source
# kimi_delta_attention_kda_gb300/csrc/kda_common.cuh.
OFF_KS, OFF_QS, OFF_KE, OFF_AKB, OFF_AQK, OFF_D = 0, 4096, 8192, 12288, 12800, 13312
PACKET_BYTES = 13824


def _sw128_index(rows):
    """Byte offsets of every BF16 element (r, c) of a [rows][128] SW128 tile."""
    r = np.arange(rows)[:, None]
    c = np.arange(128)[None, :]
    x = c // 8
    slab, chunk = x >> 3, x & 7
    return slab * rows * 128 + r * 128 + ((chunk ^ (r & 7)) << 4) + (c % 8) * 2


def _sw32_index(rows):
    r = np.arange(rows)[:, None]
    c = np.arange(16)[None, :]
    x = c // 8
    return r * 32 + ((x ^ ((r >> 2) & 1)) << 4) + (c % 8) * 2


def _bf16_at(buf, base, idx):
    """Gather BF16 values at byte offsets base + idx from a uint8 array [..., bytes]."""
    lo = buf[..., base + idx].astype(np.uint32)
    hi = buf[..., base + idx + 1].astype(np.uint32)
    bits = (lo | (hi << 8)) << 16
    return bits.view(np.float32).astype(np.float64)


def _f16_at(buf, base, idx):
    """Gather FP16 values at byte offsets base + idx from a uint8 array [..., bytes]."""
    lo = buf[..., base + idx].astype(np.uint16)
    hi = buf[..., base + idx + 1].astype(np.uint16)
    return (lo | (hi << 8)).view(np.float16).astype(np.float64)


def unpack_packets(packets):
    """Decode packets (uint8 [..., PACKET_BYTES]) into float64 arrays."""
    p = np.ascontiguousarray(packets)
    i128, i32 = _sw128_index(16), _sw32_index(16)
    iKE = _sw32_index(128)
    dp = p[..., OFF_D:OFF_D + 512].copy().view(np.float32).astype(np.float64)
    c = np.arange(128)
    d = dp[..., 16 * (c & 7) + 2 * (c >> 4) + ((c >> 3) & 1)]   # undo the permutation
    return {
        "Kprime": _bf16_at(p, OFF_KS, i128),       # -(A^kk B) K^start^T [..., 16 tokens, 128 keys]
        "Qst_s": _bf16_at(p, OFF_QS, i128),        # s * Q^start rows
        "KendT": _f16_at(p, OFF_KE, iKE),          # [..., 128 keys, 16 tokens], FP16
        "AkkB": _bf16_at(p, OFF_AKB, i32),         # A^kk with column j scaled by beta_j
        "Aqk": _f16_at(p, OFF_AQK, i32),           # FP16
        "D": d,
    }


def per_head_errors(got, ref, head_axis):
    """rel-Frobenius and max-abs error for each index of `head_axis`."""
    got = np.moveaxis(np.asarray(got, dtype=np.float64), head_axis, 0)
    ref = np.moveaxis(np.asarray(ref, dtype=np.float64), head_axis, 0)
    out = []
    for g, r in zip(got, ref):
        den = np.linalg.norm(r)
        rel = np.linalg.norm(g - r) / den if den > 0 else 0.0
        out.append((rel, float(np.abs(g - r).max()) if g.size else 0.0))
    return out


def assert_within_tolerance(got, ref, head_axis, what):
    errs = per_head_errors(got, ref, head_axis)
    for i, (rel, mx) in enumerate(errs):
        den_zero = not np.any(np.moveaxis(np.asarray(ref), head_axis, 0)[i])
        assert (den_zero or rel <= REL_FRO_TOL) and mx <= MAX_ABS_TOL, (
            "%s: head-slice %d rel-Frobenius %.3e (tol %.0e), max-abs %.3e (tol %.0e)"
            % (what, i, rel, REL_FRO_TOL, mx, MAX_ABS_TOL))
    return errs


def check_against_oracle(inp, out, final, heads=None):
    """Compare a GPU result with the oracle on the given heads (all by default).

    `inp` is a dict from kimi_delta_attention_kda_gb300.synthetic; `out` and
    `final` are CPU tensors of the GPU results.  Errors are checked per
    (sequence, head) for O and per (sequence, head) for the final state.
    """
    H = inp["q"].shape[2]
    hs = list(range(H)) if heads is None else list(heads)
    sl = lambda t: None if t is None else t[:, :, hs].contiguous()
    init = inp["init_state"]
    init_s = None if init is None else init[:, hs].contiguous()
    cu = inp["cu_seqlens"]
    o_ref, f_ref = oracle.kda_token(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["g"]),
                                    inp["beta"][:, :, hs].contiguous(), init_s,
                                    cu_seqlens=None if cu is None else cu.numpy())
    o_gpu = out[:, :, hs].double().numpy()
    f_gpu = final[:, hs].double().numpy()
    errs = {"out": [], "final": []}
    if cu is None:
        B = o_ref.shape[0]
        for b in range(B):
            errs["out"] += assert_within_tolerance(o_gpu[b], o_ref[b], 1, "O seq %d" % b)
    else:
        c = cu.numpy()
        for n in range(len(c) - 1):
            if c[n + 1] > c[n]:
                errs["out"] += assert_within_tolerance(o_gpu[0, c[n]:c[n + 1]],
                                                       o_ref[0, c[n]:c[n + 1]], 1, "O seq %d" % n)
    for n in range(f_ref.shape[0]):
        errs["final"] += assert_within_tolerance(f_gpu[n], f_ref[n], 0, "final seq %d" % n)
    return errs


def to_device(inp, device="cuda"):
    d = {}
    for key in ("q", "k", "v", "g", "beta", "init_state", "cu_seqlens"):
        t = inp[key]
        d[key] = None if t is None else t.to(device)
    return d
