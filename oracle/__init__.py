"""FP64 CPU oracle for Kimi Delta Attention (KDA) prefill.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  It shares no code with
the CUDA library in ``kimi_delta_attention_kda_gb300`` and never imports it.

The arithmetic lives in ``kda_oracle.c`` (plain C, FP64, IEEE: built with
``-ffp-contract=off`` so that x86 and Arm hosts round identically).  This
module only compiles it, converts arrays to contiguous float64 and calls it.

Functions (see ``kda_oracle.c`` for the equations and their sources):

* ``kda_token``  -- per-token gated delta rule (the chunkwise equations of
  "FlashKDA column split" section 1 taken with one-token chunks).
* ``kda_chunk``  -- the chunkwise equations of "FlashKDA column split"
  section 1 for any chunk length, with A^kk by forward substitution or by the
  Neumann product of "K3's KDA precision problem" (section "Matrix inversion in
  FlashKDA").
* ``chunk_intermediates`` -- per-chunk K^start, Q^start, K^end, D_{0:C-1},
  A^kk and A^qk.
* ``unitri_inverse`` -- (I + L)^{-1} alone.
* ``sigmoid`` -- beta from a logit (flashinfer kda_prefill, beta_is_logit);
  ``kda_token`` and ``kda_chunk`` apply it with ``beta_is_logit=True``.

Conventions: q, k, g are ``[B, T, H, dk]``, v is ``[B, T, H, dv]``, beta is
``[B, T, H]``, states are ``[N, H, dv, dk]`` (rows = value channels).  Packed
variable-length input passes ``B == 1`` and ``cu_seqlens`` (int64, N + 1).
Defaults follow the readings of the pages used throughout this project:
scale ``s = 1 / sqrt(dk)`` and L2 normalisation ``x / sqrt(sum x^2 + 1e-6)``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

L2NORM_EPS = 1e-6


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``kda_oracle.c`` (or another copy of it) into a shared library."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    D = ctypes.c_double
    I = ctypes.c_int
    lib.kda_oracle_token.argtypes = [P] * 8 + [I64] * 5 + [P, D, D, I]
    lib.kda_oracle_token.restype = I
    lib.kda_oracle_chunk.argtypes = [P] * 8 + [I64] * 5 + [P, D, D, I, I64, I]
    lib.kda_oracle_chunk.restype = I
    lib.kda_oracle_chunk_intermediates.argtypes = [P] * 10 + [I64] * 4 + [P, D, D, I, I64, I]
    lib.kda_oracle_chunk_intermediates.restype = I
    lib.kda_oracle_unitri_inverse.argtypes = [P, P, I64, I]
    lib.kda_oracle_unitri_inverse.restype = I
    lib.kda_oracle_sigmoid.argtypes = [P, P, I64]
    lib.kda_oracle_sigmoid.restype = I
    lib.kda_oracle_num_threads.argtypes = []
    lib.kda_oracle_num_threads.restype = I
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


class Variant:
    """The oracle's functions bound to another build of its source (used by
    the tests that plant mistakes in a copy of ``kda_oracle.c``)."""

    def __init__(self, lib_path):
        self._lib = _bind(lib_path)

    def kda_token(self, *a, **kw):
        return kda_token(*a, _lib=self._lib, **kw)

    def kda_chunk(self, *a, **kw):
        return kda_chunk(*a, _lib=self._lib, **kw)

    def chunk_intermediates(self, *a, **kw):
        return chunk_intermediates(*a, _lib=self._lib, **kw)

    def unitri_inverse(self, *a, **kw):
        return unitri_inverse(*a, _lib=self._lib, **kw)

    def sigmoid(self, *a, **kw):
        return sigmoid(*a, _lib=self._lib, **kw)


def num_threads() -> int:
    return int(_load().kda_oracle_num_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact widening to float64
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _geometry(q, v, cu_seqlens):
    if q.ndim != 4 or v.ndim != 4:
        raise ValueError("q and v must be [B, T, H, d]")
    B, T, H, dk = q.shape
    dv = v.shape[3]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        if B != 1:
            raise ValueError("packed input needs B == 1")
        N = int(cu.shape[0] - 1)
        return N, T, H, dk, dv, cu
    return B, T, H, dk, dv, None


def _check(rc, name):
    if rc != 0:
        raise ValueError("%s failed with status %d" % (name, rc))


def kda_token(q, k, v, g, beta, init_state=None, cu_seqlens=None, scale=None,
              eps=L2NORM_EPS, l2norm=True, want_final=True, beta_is_logit=False, _lib=None):
    """Per-token recurrence; returns ``(out [B,T,H,dv], final [N,H,dv,dk])``.
    With ``beta_is_logit`` the beta argument holds logits and the operation
    uses sigmoid(beta) (:func:`sigmoid`)."""
    lib = _lib or _load()
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    if beta_is_logit:
        beta = sigmoid(beta, _lib=lib)
    init = _f64(init_state)
    N, T, H, dk, dv, cu = _geometry(q, v, cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    out = np.zeros(v.shape, dtype=np.float64)
    final = np.zeros((N, H, dv, dk), dtype=np.float64) if want_final else None
    tokens = q.shape[0] * q.shape[1]
    rc = lib.kda_oracle_token(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init),
                              _ptr(out), _ptr(final), N, T if cu is None else tokens, H, dk,
                              dv, _ptr(cu), float(scale), float(eps), int(bool(l2norm)))
    _check(rc, "kda_oracle_token")
    return out, final


def kda_chunk(q, k, v, g, beta, init_state=None, cu_seqlens=None, scale=None,
              eps=L2NORM_EPS, l2norm=True, chunk=16, inverse="forward", beta_is_logit=False,
              _lib=None):
    """Chunkwise form; returns ``(out, final)`` like :func:`kda_token`."""
    lib = _lib or _load()
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    if beta_is_logit:
        beta = sigmoid(beta, _lib=lib)
    init = _f64(init_state)
    N, T, H, dk, dv, cu = _geometry(q, v, cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    mode = {"forward": 0, "neumann": 1}[inverse]
    out = np.zeros(v.shape, dtype=np.float64)
    final = np.zeros((N, H, dv, dk), dtype=np.float64)
    tokens = q.shape[0] * q.shape[1]
    rc = lib.kda_oracle_chunk(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init),
                              _ptr(out), _ptr(final), N, T if cu is None else tokens, H, dk,
                              dv, _ptr(cu), float(scale), float(eps), int(bool(l2norm)),
                              int(chunk), mode)
    _check(rc, "kda_oracle_chunk")
    return out, final


def chunk_offsets(lengths, chunk=16):
    """First chunk index of every sequence (length N + 1) for the given lengths."""
    first = [0]
    for n in lengths:
        first.append(first[-1] + (int(n) + chunk - 1) // chunk)
    return first


def chunk_intermediates(q, k, g, beta, cu_seqlens=None, scale=None, eps=L2NORM_EPS,
                        l2norm=True, chunk=16, inverse="forward", _lib=None):
    """Per-(chunk, head) K^start, Q^start, K^end, D, A^kk, A^qk as a dict of arrays.

    Chunks are numbered sequence by sequence; arrays have a leading
    ``[n_chunks, H]`` pair of dimensions.
    """
    lib = _lib or _load()
    q, k, g, beta = map(_f64, (q, k, g, beta))
    B, T, H, dk = q.shape
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        N = int(cu.shape[0] - 1)
        lengths = np.diff(cu)
        Tt = q.shape[1]
    else:
        cu = None
        N = B
        lengths = [T] * B
        Tt = T
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    nch = chunk_offsets(lengths, chunk)[-1]
    C = chunk
    out = {
        "Kst": np.zeros((nch, H, C, dk)), "Qst": np.zeros((nch, H, C, dk)),
        "Kend": np.zeros((nch, H, C, dk)), "D": np.zeros((nch, H, dk)),
        "Akk": np.zeros((nch, H, C, C)), "Aqk": np.zeros((nch, H, C, C)),
    }
    mode = {"forward": 0, "neumann": 1}[inverse]
    rc = lib.kda_oracle_chunk_intermediates(
        _ptr(q), _ptr(k), _ptr(g), _ptr(beta), _ptr(out["Kst"]), _ptr(out["Qst"]),
        _ptr(out["Kend"]), _ptr(out["D"]), _ptr(out["Akk"]), _ptr(out["Aqk"]), N, Tt, H, dk,
        _ptr(cu), float(scale), float(eps), int(bool(l2norm)), int(chunk), mode)
    _check(rc, "kda_oracle_chunk_intermediates")
    return out


def unitri_inverse(L, mode="forward", _lib=None):
    """(I + L)^{-1} for a strictly lower-triangular square matrix L."""
    lib = _lib or _load()
    L = _f64(L)
    C = L.shape[0]
    X = np.zeros_like(L)
    rc = lib.kda_oracle_unitri_inverse(_ptr(L), _ptr(X), C, {"forward": 0, "neumann": 1}[mode])
    _check(rc, "kda_oracle_unitri_inverse")
    return X


def sigmoid(x, _lib=None):
    """Elementwise 1 / (1 + exp(-x)) in FP64 (beta from a logit, flashinfer
    kda_prefill "Optimized Blackwell prefill subset", beta_is_logit)."""
    lib = _lib or _load()
    x = _f64(x)
    y = np.zeros_like(x)
    _check(lib.kda_oracle_sigmoid(_ptr(x), _ptr(y), int(x.size)), "kda_oracle_sigmoid")
    return y
