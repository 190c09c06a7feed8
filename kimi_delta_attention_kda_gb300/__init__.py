"""GB300-native Kimi Delta Attention (KDA) prefill.

The operation runs in ``libkda.so`` (CUDA kernels for sm_103a behind the C ABI
of ``include/kda.h``).  This package only builds that library and marshals
PyTorch tensors into its entry points; PyTorch provides device memory and
streams.  There is no CPU path.
"""

from __future__ import annotations

from . import _lib
from ._lib import (KdaError, auto_split, device_status, packet_bytes, plan_fused,
                   plan_long_split, plan_segments, set_engine, set_fusion, set_segments,
                   set_split, workspace_bytes)

HEAD_DIM = 128

__all__ = ["kda_prefill", "kda_prefill_host", "prep_only", "KdaError", "device_status", "set_split", "set_engine",
           "set_fusion", "plan_fused", "plan_long_split", "set_segments", "plan_segments",
           "auto_split",
           "workspace_bytes", "packet_bytes", "HEAD_DIM"]


def _require(cond, msg):
    if not cond:
        raise ValueError(msg)


def _ptr(t):
    return 0 if t is None else int(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def kda_prefill(q, k, v, g, beta, init_state=None, cu_seqlens=None, out=None,
                final_state=None, output_final_state=True, stream=None,
                checkpoint_every_n_tokens=None, state_checkpoints=None,
                checkpoint_cu_starts=None, beta_is_logit=False):
    """KDA prefill on CUDA tensors; returns ``(out, final_state)``, or
    ``(out, final_state, state_checkpoints)`` with checkpoints.

    q, k, v: bf16 ``[B, T, H, 128]``; g: fp32 ``[B, T, H, 128]`` (log-decay in
    [-5, 0]); beta: bf16 ``[B, T, H]``; init_state: bf16 ``[N, H, 128, 128]`` or
    None; cu_seqlens: int64 ``[N + 1]`` on the device for the packed layout
    (then ``B == 1``).  ``final_state`` may be ``init_state`` for an in-place
    update.  With ``checkpoint_every_n_tokens`` (a positive multiple of 16),
    ``state_checkpoints`` (bf16 ``[C, H, 128, 128]``) receives the state before
    every interval of each sequence at rows ``checkpoint_cu_starts[n]`` ..
    (int64 ``[N + 1]`` on the device; see ``kda_prefill_checkpointed`` in
    include/kda.h).  With ``beta_is_logit`` beta holds logits and the
    operation uses sigmoid(beta) (``kda_prefill_ex``).  The call is
    asynchronous on ``stream`` (default: the current PyTorch stream).
    """
    import torch
    _require(q.dim() == 4 and q.shape[-1] == HEAD_DIM, "q must be [B, T, H, 128]")
    B, T, H, _ = q.shape
    for name, t in (("k", k), ("v", v)):
        _require(t.shape == q.shape, "%s must have the shape of q" % name)
    _require(g.shape == q.shape, "g must have the shape of q")
    _require(beta.shape == q.shape[:3], "beta must be [B, T, H]")
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("g", g, torch.float32),
                        ("beta", beta, torch.bfloat16)):
        _require(t.is_cuda and t.dtype == dt and t.is_contiguous(),
                 "%s must be a contiguous %s CUDA tensor" % (name, dt))
    if cu_seqlens is not None:
        _require(B == 1, "packed input needs B == 1")
        _require(cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int64 and cu_seqlens.dim() == 1
                 and cu_seqlens.is_contiguous(), "cu_seqlens must be a contiguous int64 CUDA vector")
        N = cu_seqlens.numel() - 1
        n_arg = N
    else:
        N = B
        n_arg = B
    if init_state is not None:
        _require(init_state.is_cuda and init_state.dtype == torch.bfloat16
                 and init_state.is_contiguous()
                 and tuple(init_state.shape) == (N, H, HEAD_DIM, HEAD_DIM),
                 "init_state must be a contiguous bf16 [N, H, 128, 128] CUDA tensor")
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, HEAD_DIM, HEAD_DIM), dtype=torch.bfloat16,
                                  device=q.device)
    flags = _lib.FLAG_BETA_LOGIT if beta_is_logit else 0
    if checkpoint_every_n_tokens is None and flags:
        rc = _lib.prefill_ex_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
                                 _ptr(out), _ptr(final_state), n_arg, T, H, _ptr(cu_seqlens),
                                 flags, 0, 0, 0, 0, _stream_handle(stream))
        if rc != 0:
            raise KdaError(rc, "kda_prefill_ex")
        return out, final_state
    if checkpoint_every_n_tokens is None:
        rc = _lib.prefill_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
                              _ptr(out), _ptr(final_state), n_arg, T, H, _ptr(cu_seqlens),
                              _stream_handle(stream))
        if rc != 0:
            raise KdaError(rc, "kda_prefill")
        return out, final_state
    _require(state_checkpoints is not None and checkpoint_cu_starts is not None,
             "checkpoints need state_checkpoints and checkpoint_cu_starts")
    _require(state_checkpoints.is_cuda and state_checkpoints.dtype == torch.bfloat16
             and state_checkpoints.is_contiguous() and state_checkpoints.dim() == 4
             and tuple(state_checkpoints.shape[1:]) == (H, HEAD_DIM, HEAD_DIM),
             "state_checkpoints must be a contiguous bf16 [C, H, 128, 128] CUDA tensor")
    _require(checkpoint_cu_starts.is_cuda and checkpoint_cu_starts.dtype == torch.int64
             and checkpoint_cu_starts.is_contiguous() and checkpoint_cu_starts.numel() == N + 1,
             "checkpoint_cu_starts must be a contiguous int64 [N + 1] CUDA vector")
    if flags:
        rc = _lib.prefill_ex_raw(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state), _ptr(out),
            _ptr(final_state), n_arg, T, H, _ptr(cu_seqlens), flags, checkpoint_every_n_tokens,
            _ptr(state_checkpoints), _ptr(checkpoint_cu_starts), state_checkpoints.shape[0],
            _stream_handle(stream))
    else:
        rc = _lib.prefill_checkpointed_raw(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state), _ptr(out),
            _ptr(final_state), n_arg, T, H, _ptr(cu_seqlens), checkpoint_every_n_tokens,
            _ptr(state_checkpoints), _ptr(checkpoint_cu_starts), state_checkpoints.shape[0],
            _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_prefill_ex" if flags else "kda_prefill_checkpointed")
    return out, final_state, state_checkpoints


def kda_prefill_host(q, k, v, g, beta, init_state=None, cu_seqlens=None, out=None,
                     final_state=None, output_final_state=True, stream=None):
    """KDA prefill on CPU (host) tensors through ``kda_prefill_host``: the
    library copies the inputs to the current CUDA device, computes, and copies
    ``out`` and ``final_state`` back, overlapping the copies with the work.
    Shapes and dtypes as ``kda_prefill``; every tensor (cu_seqlens included)
    is a contiguous CPU tensor, pinned for asynchronous, overlapped copies
    (``tensor.pin_memory()``).  New outputs are allocated pinned.  The call is
    asynchronous on ``stream``: synchronise it before reading the outputs.
    Returns ``(out, final_state)``."""
    import torch
    _require(q.dim() == 4 and q.shape[-1] == HEAD_DIM, "q must be [B, T, H, 128]")
    B, T, H, _ = q.shape
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("g", g, torch.float32),
                        ("beta", beta, torch.bfloat16)):
        _require(not t.is_cuda and t.dtype == dt and t.is_contiguous(),
                 "%s must be a contiguous %s CPU tensor" % (name, dt))
    for name, t in (("k", k), ("v", v), ("g", g)):
        _require(t.shape == q.shape, "%s must have the shape of q" % name)
    _require(beta.shape == q.shape[:3], "beta must be [B, T, H]")
    if cu_seqlens is not None:
        _require(B == 1, "packed input needs B == 1")
        _require(not cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int64
                 and cu_seqlens.dim() == 1 and cu_seqlens.is_contiguous(),
                 "cu_seqlens must be a contiguous int64 CPU vector")
        N = n_arg = cu_seqlens.numel() - 1
    else:
        N = n_arg = B
    if init_state is not None:
        _require(not init_state.is_cuda and init_state.dtype == torch.bfloat16
                 and init_state.is_contiguous()
                 and tuple(init_state.shape) == (N, H, HEAD_DIM, HEAD_DIM),
                 "init_state must be a contiguous bf16 [N, H, 128, 128] CPU tensor")
    if out is None:
        out = torch.empty(v.shape, dtype=torch.bfloat16).pin_memory()
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, HEAD_DIM, HEAD_DIM), dtype=torch.bfloat16).pin_memory()
    for name, t in (("out", out), ("final_state", final_state)):
        if t is not None:
            _require(not t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous(),
                     "%s must be a contiguous bf16 CPU tensor" % name)
    rc = _lib.prefill_host_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
                               _ptr(out), _ptr(final_state), n_arg, T, H, _ptr(cu_seqlens),
                               _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_prefill_host")
    return out, final_state


def prep_only(q, k, g, beta, cu_seqlens=None, stream=None):
    """Run only the chunk preparation; returns the raw packets as a uint8 tensor
    of shape ``[n_chunks_upper_bound, H, packet_bytes]``."""
    import torch
    B, T, H, _ = q.shape
    packed = cu_seqlens is not None
    n_arg = cu_seqlens.numel() - 1 if packed else B
    nbytes = _lib.workspace_bytes(n_arg, T, H, packed)
    pb = packet_bytes()
    meta = 0
    if packed:
        meta = 256 + ((8 * (n_arg + 1) + 255) // 256) * 256
    n_chunk_heads = (nbytes - meta) // pb
    packets = torch.zeros((n_chunk_heads // H, H, pb), dtype=torch.uint8, device=q.device)
    rc = _lib.prep_only_raw(_ptr(q), _ptr(k), _ptr(g), _ptr(beta), n_arg, T, H, _ptr(cu_seqlens),
                            _ptr(packets), packets.numel(), _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_prep_only")
    return packets
