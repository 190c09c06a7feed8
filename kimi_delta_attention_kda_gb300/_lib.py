"""ctypes binding of ``libkda.so`` (the C ABI declared in ``include/kda.h``).

Argument marshalling only: every step of the operation runs in the library's
CUDA kernels.  There is no fallback: if the library is missing or cannot be
loaded, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")

KDA_OK = 0
KDA_DEV_BAD_SEQLENS = 1
KDA_DEV_PIPE_TIMEOUT = 2

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (where, error_string(status), status))


def load():
    """Load ``libkda.so`` (built by ``kimi_delta_attention_kda_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libkda.so is not built (run kimi_delta_attention_kda_gb300.build"
                               ".build() or __graft_entry__.build())")
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.kda_prefill.argtypes = [P] * 8 + [I64] * 3 + [P, P]
        lib.kda_prefill.restype = I
        lib.kda_prefill_checkpointed.argtypes = [P] * 8 + [I64] * 3 + [P, I64, P, P, I64, P]
        lib.kda_prefill_checkpointed.restype = I
        lib.kda_prefill_ex.argtypes = [P] * 8 + [I64] * 3 + [P, ctypes.c_uint32, I64, P, P, I64, P]
        lib.kda_prefill_ex.restype = I
        lib.kda_error_string.argtypes = [I]
        lib.kda_error_string.restype = ctypes.c_char_p
        lib.kda_device_status.argtypes = [P, ctypes.POINTER(I)]
        lib.kda_device_status.restype = I
        lib.kda_set_split.argtypes = [I]
        lib.kda_set_split.restype = I
        lib.kda_set_engine.argtypes = [I]
        lib.kda_set_engine.restype = I
        lib.kda_set_fusion.argtypes = [I]
        lib.kda_set_fusion.restype = I
        lib.kda_set_segments.argtypes = [I, I64]
        lib.kda_set_segments.restype = I
        lib.kda_plan_segments.argtypes = [I64, I64, I64, I, ctypes.POINTER(I64)]
        lib.kda_plan_segments.restype = I
        lib.kda_plan_fused.argtypes = [I64, I64, I64, I, ctypes.POINTER(I)]
        lib.kda_plan_fused.restype = I
        lib.kda_plan_long_split.argtypes = [I64, I64, I64, ctypes.POINTER(I64)]
        lib.kda_plan_long_split.restype = I
        lib.kda_auto_split.argtypes = [I64, I64, ctypes.POINTER(I)]
        lib.kda_auto_split.restype = I
        lib.kda_workspace_bytes.argtypes = [I64, I64, I64, I, ctypes.POINTER(I64)]
        lib.kda_workspace_bytes.restype = I
        lib.kda_prep_only.argtypes = [P] * 4 + [I64] * 3 + [P, P, I64, P]
        lib.kda_prep_only.restype = I
        lib.kda_packet_bytes.argtypes = []
        lib.kda_packet_bytes.restype = I64
        lib.kda_profile_begin.argtypes = [I]
        lib.kda_profile_begin.restype = I
        D = ctypes.POINTER(ctypes.c_double)
        lib.kda_profile_end.argtypes = [D, D, ctypes.POINTER(I)]
        lib.kda_profile_end.restype = I
        lib.kda_profile_end_detail.argtypes = [D, ctypes.POINTER(I)]
        lib.kda_profile_end_detail.restype = I
        lib.kda_chain_step_ns.argtypes = [ctypes.POINTER(ctypes.c_double)]
        lib.kda_chain_step_ns.restype = I
        lib.kda_set_host_pieces.argtypes = [I]
        lib.kda_set_host_pieces.restype = I
        lib.kda_last_call_launches.argtypes = [ctypes.POINTER(I64)]
        lib.kda_last_call_launches.restype = I
        lib.kda_prefill_host.argtypes = [P] * 8 + [I64] * 3 + [P, P]
        lib.kda_prefill_host.restype = I
        lib.kda_prefill_noalloc.argtypes = [P] * 8 + [I64] * 3 + [P, P]
        lib.kda_prefill_noalloc.restype = I
        lib.kda_noalloc_scratch_bytes.argtypes = []
        lib.kda_noalloc_scratch_bytes.restype = I64
        _lib = lib
        return lib


def error_string(status: int) -> str:
    try:
        return load().kda_error_string(int(status)).decode()
    except Exception:  # library missing: still give a readable message
        return "status %d" % status


def _check(rc: int, where: str):
    if rc != KDA_OK:
        raise KdaError(rc, where)


def prefill_raw(q, k, v, g, beta, init_state, out, final_state, B, T, H, cu_seqlens, stream):
    """Call ``kda_prefill`` with integer device addresses (0 for NULL); returns the status."""
    return load().kda_prefill(q or None, k or None, v or None, g or None, beta or None,
                              init_state or None, out or None, final_state or None,
                              int(B), int(T), int(H), cu_seqlens or None, stream or None)


def set_host_pieces(n):
    """Pieces kda_prefill_host cuts a call into (0: automatic)."""
    rc = load().kda_set_host_pieces(int(n))
    if rc != 0:
        raise KdaError(rc, "kda_set_host_pieces")


def last_call_launches():
    """Kernels the last kda_prefill / kda_prefill_host call of this thread enqueued."""
    n = ctypes.c_int64(0)
    rc = load().kda_last_call_launches(ctypes.byref(n))
    if rc != 0:
        raise KdaError(rc, "kda_last_call_launches")
    return n.value


def prefill_host_raw(q, k, v, g, beta, init_state, out, final_state, B, T, H, cu_seqlens, stream):
    """Call ``kda_prefill_host`` with integer HOST addresses (0 for NULL); returns the status."""
    return load().kda_prefill_host(q or None, k or None, v or None, g or None, beta or None,
                                   init_state or None, out or None, final_state or None,
                                   int(B), int(T), int(H), cu_seqlens or None, stream or None)


def prefill_checkpointed_raw(q, k, v, g, beta, init_state, out, final_state, B, T, H, cu_seqlens,
                             every, states, cu_starts, rows, stream):
    """Call ``kda_prefill_checkpointed`` with integer device addresses (0 for NULL)."""
    return load().kda_prefill_checkpointed(
        q or None, k or None, v or None, g or None, beta or None, init_state or None, out or None,
        final_state or None, int(B), int(T), int(H), cu_seqlens or None, int(every),
        states or None, cu_starts or None, int(rows), stream or None)


FLAG_BETA_LOGIT = 1


def prefill_ex_raw(q, k, v, g, beta, init_state, out, final_state, B, T, H, cu_seqlens, flags,
                   every, states, cu_starts, rows, stream):
    """Call ``kda_prefill_ex`` with integer device addresses (0 for NULL)."""
    return load().kda_prefill_ex(
        q or None, k or None, v or None, g or None, beta or None, init_state or None, out or None,
        final_state or None, int(B), int(T), int(H), cu_seqlens or None, int(flags), int(every),
        states or None, cu_starts or None, int(rows), stream or None)


def device_status(stream=0) -> int:
    st = ctypes.c_int(0)
    _check(load().kda_device_status(stream or None, ctypes.byref(st)), "kda_device_status")
    return st.value


def set_split(nsplit: int):
    _check(load().kda_set_split(int(nsplit)), "kda_set_split")


def set_engine(engine: int):
    """0 automatic, 1 column-split warp-MMA kernel, 2 tcgen05 kernel."""
    _check(load().kda_set_engine(int(engine)), "kda_set_engine")


def set_fusion(on: bool):
    """Allow (True, the default) or forbid preparation and recurrence as one launch."""
    _check(load().kda_set_fusion(1 if on else 0), "kda_set_fusion")


def set_segments(on: bool, seg_chunks: int = 0):
    """Allow (True, the default) or forbid the segmented scan over chunks;
    seg_chunks > 0 forces segments of that many chunks on every eligible call."""
    _check(load().kda_set_segments(1 if on else 0, int(seg_chunks)), "kda_set_segments")


def plan_segments(B: int, T: int, H: int, packed: bool) -> int:
    """Segments per sequence kda_prefill uses for this shape (0: serial chain)."""
    out = ctypes.c_int64(0)
    _check(load().kda_plan_segments(int(B), int(T), int(H), 1 if packed else 0, ctypes.byref(out)),
           "kda_plan_segments")
    return int(out.value)


def plan_fused(B: int, T: int, H: int, packed: bool) -> bool:
    """Whether kda_prefill runs this shape as one launch on the current device."""
    out = ctypes.c_int(0)
    _check(load().kda_plan_fused(int(B), int(T), int(H), 1 if packed else 0, ctypes.byref(out)),
           "kda_plan_fused")
    return bool(out.value)


def plan_long_split(n_seqs: int, T: int, H: int) -> int:
    """How many longest sequences of a packed call run at split 2 in a second
    launch (0 under the many-head one-launch form)."""
    out = ctypes.c_int64(0)
    _check(load().kda_plan_long_split(int(n_seqs), int(T), int(H), ctypes.byref(out)),
           "kda_plan_long_split")
    return int(out.value)


def auto_split(n_seqs: int, H: int) -> int:
    ns = ctypes.c_int(0)
    _check(load().kda_auto_split(int(n_seqs), int(H), ctypes.byref(ns)), "kda_auto_split")
    return ns.value


def workspace_bytes(B: int, T: int, H: int, packed: bool) -> int:
    b = ctypes.c_int64(0)
    _check(load().kda_workspace_bytes(int(B), int(T), int(H), int(bool(packed)), ctypes.byref(b)),
           "kda_workspace_bytes")
    return b.value


def packet_bytes() -> int:
    return int(load().kda_packet_bytes())


def prep_only_raw(q, k, g, beta, B, T, H, cu_seqlens, packets, packets_bytes, stream):
    return load().kda_prep_only(q or None, k or None, g or None, beta or None, int(B), int(T),
                                int(H), cu_seqlens or None, packets or None, int(packets_bytes),
                                stream or None)


def profile_begin(max_calls: int):
    _check(load().kda_profile_begin(int(max_calls)), "kda_profile_begin")


def profile_end():
    """Returns (prep_ms_total, recurrence_ms_total, calls)."""
    p, r, n = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_int(0)
    _check(load().kda_profile_end(ctypes.byref(p), ctypes.byref(r), ctypes.byref(n)),
           "kda_profile_end")
    return p.value, r.value, n.value


def profile_end_detail():
    """Returns ([prep, transition, segment chain, recurrence] ms totals, calls)."""
    t = (ctypes.c_double * 4)()
    n = ctypes.c_int(0)
    _check(load().kda_profile_end_detail(t, ctypes.byref(n)), "kda_profile_end_detail")
    return [t[i] for i in range(4)], n.value


def chain_step_ns() -> float:
    """Nanoseconds per step of the shortest dependent chunk-step chain (one warp)."""
    v = ctypes.c_double(0)
    _check(load().kda_chain_step_ns(ctypes.byref(v)), "kda_chain_step_ns")
    return v.value


def prefill_noalloc_raw(q, k, v, g, beta, init_state, out, final_state, B, T, H, cu_seqlens,
                        stream):
    """Call ``kda_prefill_noalloc`` (no allocation; fixed in-library scratch) with
    integer device addresses (0 for NULL); returns the status."""
    return load().kda_prefill_noalloc(q or None, k or None, v or None, g or None, beta or None,
                                      init_state or None, out or None, final_state or None,
                                      int(B), int(T), int(H), cu_seqlens or None, stream or None)


def noalloc_scratch_bytes() -> int:
    return int(load().kda_noalloc_scratch_bytes())
