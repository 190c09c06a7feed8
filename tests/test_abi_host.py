"""Host-side tests of the C ABI (no GPU needed).

The library must load and export every function that include/kda.h
declares, and kda_prefill must refuse bad arguments on the host, before any
CUDA call, with the documented codes.  The addresses passed here are never
dereferenced: validation runs before the library touches the device.
"""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from kimi_delta_attention_kda_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(kda_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("kda_prefill", "kda_error_string", "kda_device_status", "kda_set_split"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), "libkda.so does not export %s" % name


def test_error_strings(lib):
    for code in range(0, -10, -1):
        s = lib.kda_error_string(code).decode()
        assert s and s != "unknown KDA status"
    assert lib.kda_error_string(-99).decode() == "unknown KDA status"


A = 1 << 20       # fake, 16-byte aligned, never dereferenced
GB = 1 << 32


def call(lib, q=A, k=A + GB, v=A + 2 * GB, g=A + 3 * GB, beta=A + 4 * GB, init=0,
         out=A + 5 * GB, final=0, B=1, T=16, H=1, cu=0):
    return _lib.prefill_raw(q, k, v, g, beta, init, out, final, B, T, H, cu, 0)


def test_null_pointers(lib):
    assert call(lib, q=0) == -1
    assert call(lib, out=0) == -1
    assert call(lib, beta=0) == -1
    # with no tokens the token tensors may be NULL: validation passes and the
    # call goes on to the device query
    import torch
    if not torch.cuda.is_available():
        assert call(lib, q=0, k=0, v=0, g=0, beta=0, out=0, T=0) == -5


def test_bad_shapes(lib):
    assert call(lib, B=0) == -2
    assert call(lib, H=0) == -2
    assert call(lib, T=-1) == -2
    assert call(lib, B=1 << 40, T=1 << 40) == -2


def test_misaligned(lib):
    assert call(lib, q=A + 2) == -3
    assert call(lib, g=A + 3 * GB + 8) == -3
    assert call(lib, beta=A + 4 * GB + 1) == -3
    assert call(lib, init=A + 6 * GB + 4) == -3
    assert call(lib, cu=A + 7 * GB + 4) == -3


def test_overlaps(lib):
    # out overlapping q
    assert call(lib, out=A + 64) == -4
    # final state overlapping an input
    assert call(lib, final=A + 3 * GB + 16) == -4
    # final partially overlapping init (identical pointers are allowed)
    assert call(lib, init=A + 6 * GB, final=A + 6 * GB + 1024) == -4


def test_no_device_here(lib):
    """Valid arguments reach the device query; without a GPU that is KDA_ERR_DEVICE."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call(lib) == -5
    st = ctypes.c_int(0)
    assert lib.kda_device_status(None, ctypes.byref(st)) == -5
    ns = ctypes.c_double(0)
    assert lib.kda_chain_step_ns(ctypes.byref(ns)) == -5
    assert lib.kda_chain_step_ns(None) == -1


def test_split_option(lib):
    for ns in (0, 1, 2, 4, 8, 16):
        assert lib.kda_set_split(ns) == 0
    for ns in (3, 5, 32, -1):
        assert lib.kda_set_split(ns) == -7
    assert lib.kda_set_split(0) == 0


def test_segments_option(lib):
    for on, L in ((0, 0), (1, 0), (1, 1), (1, 64), (0, 5)):
        assert lib.kda_set_segments(on, L) == 0
    for on, L in ((2, 0), (-1, 0), (1, -1), (1, (1 << 26) + 1)):
        assert lib.kda_set_segments(on, L) == -7
    assert lib.kda_set_segments(1, 0) == 0


def test_workspace_bytes(lib):
    pb = _lib.packet_bytes()
    assert pb == 13824
    # fixed: ceil(T/16) chunks per sequence
    # packets, plus 256-aligned ready flags (one per chunk and head, and one word
    # more: the item counter of the many-head form) for a fused launch
    assert _lib.workspace_bytes(2, 40, 3, False) == 2 * 3 * 3 * pb + 256
    assert _lib.workspace_bytes(1, 0, 5, False) == 0
    # packed: (T + 15 N) // 16 chunks at most, plus the metadata block (valid
    # flag, chunk offsets and, for up to 1024 sequences, their longest-first order)
    n, T, H = 4, 100, 2
    meta = 256 + ((8 * (n + 1) + 255) // 256) * 256 + ((4 * n + 255) // 256) * 256
    assert _lib.workspace_bytes(n, T, H, True) == meta + ((T + 15 * n) // 16) * H * pb
    # fixed, few heads, long sequence: the segmented scan's three state buffers
    # as planned for a 152-SM device (B=1, H=6, T=8192: 25 segments of 21 chunks)
    import torch
    if not torch.cuda.is_available():
        st = 25 * 6 * 128 * 128 * 2
        assert _lib.workspace_bytes(1, 8192, 6, False) == 512 * 6 * pb + 12544 + 3 * st
        lib.kda_set_segments(0, 0)
        assert _lib.workspace_bytes(1, 8192, 6, False) == 512 * 6 * pb + 12544
        lib.kda_set_segments(1, 0)
        # packed, 8 sequences, 24,672 tokens, 12 heads: the many-head one-launch
        # form, so also the ready flags (and the item counter), the chunk
        # order, 4 bytes a chunk (1,549 chunks at most), and a flag a sequence
        n, T, H = 8, 24672, 12
        meta = 256 + 256 + 256
        cub = (T + 15 * n) // 16
        ready = ((cub * H * 4 + 4 + 255) // 256) * 256
        order = ((cub * 4 + 255) // 256) * 256 + 256
        assert _lib.workspace_bytes(n, T, H, True) == meta + cub * H * pb + ready + order
        lib.kda_set_fusion(0)
        assert _lib.workspace_bytes(n, T, H, True) == meta + cub * H * pb
        lib.kda_set_fusion(1)


def call_ck(lib, every=64, states=A + 9 * GB, cu_starts=A + 10 * GB, rows=4, **kw):
    args = dict(q=A, k=A + GB, v=A + 2 * GB, g=A + 3 * GB, beta=A + 4 * GB, init=0,
                out=A + 5 * GB, final=0, B=1, T=16, H=1, cu=0)
    args.update(kw)
    return _lib.prefill_checkpointed_raw(args["q"], args["k"], args["v"], args["g"], args["beta"],
                                         args["init"], args["out"], args["final"], args["B"],
                                         args["T"], args["H"], args["cu"], every, states,
                                         cu_starts, rows, 0)


def test_checkpoint_arguments(lib):
    """Checked on the host before anything launches (no GPU needed)."""
    for every in (0, -16, 8, 24, 100):
        assert call_ck(lib, every=every) == -7       # not a positive multiple of 16
    assert call_ck(lib, rows=-1) == -7
    assert call_ck(lib, cu_starts=0) == -1
    assert call_ck(lib, states=0) == -1
    assert call_ck(lib, states=A + 9 * GB + 8) == -3   # 16-byte alignment
    assert call_ck(lib, cu_starts=A + 10 * GB + 4) == -3
    # the checkpoint buffer must not overlap an input, an output or its offsets
    assert call_ck(lib, states=A + 64) == -4                      # q
    assert call_ck(lib, states=A + 5 * GB) == -4                  # out
    assert call_ck(lib, states=A + 10 * GB - 1024) == -4          # the offsets
    assert call_ck(lib, B=0) == -2                                # ordinary shape checks still apply


def test_fast_divider_matches_integer_division(tmp_path):
    """The launch-time divider of the preparation's item decoding (a
    multiply-high division, kda_prep_impl.cuh) against exact integer division at
    its hardest numerators, through its host instantiation."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "fastdiv_check")
    src = os.path.join(ROOT, "tests", "fastdiv_check.cu")
    inc = os.path.join(ROOT, "kimi_delta_attention_kda_gb300", "csrc")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-I", inc, src, "-o", exe], check=True,
                   capture_output=True, timeout=300)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout


def call_host(lib, cu=None, B=1, T=16, H=1, q=A, out=A + 5 * GB, final=0, init=0):
    """kda_prefill_host with fake host addresses (never dereferenced before
    the device query) and, for the packed layout, a real host offsets array."""
    import numpy as np
    cu_arr = None if cu is None else np.ascontiguousarray(np.asarray(cu, dtype=np.int64))
    cu_ptr = 0 if cu_arr is None else cu_arr.ctypes.data
    return _lib.prefill_host_raw(q, A + GB, A + 2 * GB, A + 3 * GB, A + 4 * GB, init, out, final,
                                 B, T, H, cu_ptr, 0)


def test_host_entry_checks_offsets_on_the_host(lib):
    """kda_prefill_host reads its HOST cu_seqlens before anything else and
    refuses a broken contract with KDA_ERR_SEQLENS (-9)."""
    assert call_host(lib, cu=[1, 16], B=1, T=16) == -9        # cu[0] != 0
    assert call_host(lib, cu=[0, 32, 16], B=2, T=16) == -9    # decreasing
    assert call_host(lib, cu=[0, 16, 40], B=2, T=48) == -9    # cu[N] != T
    assert call_host(lib, B=0) == -2
    assert call_host(lib, q=0) == -1
    assert call_host(lib, out=A + 64) == -4                   # host out overlaps host q
    import torch
    if not torch.cuda.is_available():
        # valid arguments (no alignment rule for host buffers) reach the device query
        assert call_host(lib, cu=[0, 0, 16, 48], B=3, T=48) == -5
        assert call_host(lib, q=A + 2) == -5


def test_huge_head_count_is_a_shape_error_not_a_crash(lib):
    """With no tokens and H = 2^50, H * 128 * 128 wraps to zero in 64 bits; every
    entry point must refuse the shape (KDA_ERR_SHAPE) before dividing by it."""
    H = 1 << 50
    assert call(lib, T=0, H=H) == -2
    assert call(lib, T=0, H=H, cu=A + 7 * GB) == -2
    assert call_ck(lib, T=0, H=H) == -2
    assert call_host(lib, T=0, H=H) == -2
    assert _lib.prefill_noalloc_raw(A, A + GB, A + 2 * GB, A + 3 * GB, A + 4 * GB, 0,
                                    A + 5 * GB, 0, 1, 0, H, 0, 0) == -2
    assert _lib.prep_only_raw(A, A + GB, A + 3 * GB, A + 4 * GB, 1, 0, H, 0, A + 5 * GB,
                              1 << 40, 0) == -2
    n = ctypes.c_int64(0)
    flag = ctypes.c_int(0)
    assert lib.kda_workspace_bytes(1, 0, H, 0, ctypes.byref(n)) == -2
    assert lib.kda_plan_segments(1, 0, H, 0, ctypes.byref(n)) == -2
    assert lib.kda_plan_fused(1, 0, H, 0, ctypes.byref(flag)) == -2
    assert lib.kda_plan_long_split(1, 0, H, ctypes.byref(n)) == -2


def call_noalloc(lib, B=1, T=16, H=1, cu=0):
    return _lib.prefill_noalloc_raw(A, A + GB, A + 2 * GB, A + 3 * GB, A + 4 * GB, 0,
                                    A + 5 * GB, 0, B, T, H, cu, 0)


def test_noalloc_scratch_boundary(lib):
    """kda_prefill_noalloc's fixed 48 MiB scratch holds 3,640 packets of 13,824
    bytes plus 12,288 bytes.  The refusal (KDA_ERR_SCRATCH) is decided on the
    host before any device work; a shape that fits goes on to the device
    query (KDA_ERR_DEVICE here, with no GPU)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: shapes that fit would launch on fake pointers")
    cap = 48 << 20
    assert _lib.noalloc_scratch_bytes() == cap
    assert cap // 13824 == 3640 and cap - 3640 * 13824 == 12288
    # fixed layout: 3,640 chunks of one head fit exactly, one more does not
    assert call_noalloc(lib, T=3640 * 16) == -5
    assert call_noalloc(lib, T=3640 * 16 + 1) == -8
    assert call_noalloc(lib, T=1820 * 16, H=2) == -5
    assert call_noalloc(lib, T=1820 * 16 + 1, H=2) == -8
    # packed: chunk bound (T + 15 N) // 16 and 256 + ceil(8 (N + 1) / 256) * 256
    # bytes of metadata.  N = 1503 sequences: 3,640 packets + 12,288 bytes of
    # metadata fill the array to the byte; N = 1504: the packets still fit but
    # the metadata (12,544 bytes) does not.
    def need(N, T):
        return 256 + -(-8 * (N + 1) // 256) * 256 + (T + 15 * N) // 16 * 13824
    assert need(1503, 35695) == cap
    assert call_noalloc(lib, B=1503, T=35695, cu=A + 7 * GB) == -5
    assert (35695 + 15 * 1504) // 16 * 13824 <= cap < need(1504, 35695)
    assert call_noalloc(lib, B=1504, T=35695, cu=A + 7 * GB) == -8


def test_prefill_ex_arguments(lib):
    """kda_prefill_ex: unknown flag bits are KDA_ERR_ARG; its checkpoint
    arguments are checked like kda_prefill_checkpointed's (host only)."""
    def ex(flags=1, every=0, states=0, cu_starts=0, rows=0, **kw):
        a = dict(q=A, k=A + GB, v=A + 2 * GB, g=A + 3 * GB, beta=A + 4 * GB, init=0,
                 out=A + 5 * GB, final=0, B=1, T=16, H=1, cu=0)
        a.update(kw)
        return _lib.prefill_ex_raw(a["q"], a["k"], a["v"], a["g"], a["beta"], a["init"], a["out"],
                                   a["final"], a["B"], a["T"], a["H"], a["cu"], flags, every,
                                   states, cu_starts, rows, 0)
    for flags in (2, 4, 3, 1 << 31):
        assert ex(flags=flags) == -7
    assert ex(flags=1, B=0) == -2
    assert ex(flags=1, q=0) == -1
    assert ex(flags=1, states=A + 9 * GB, cu_starts=A + 10 * GB, every=8, rows=4) == -7
    assert ex(flags=1, states=A + 9 * GB, cu_starts=0, every=16, rows=4) == -1
    assert ex(flags=1, states=A + 9 * GB + 8, cu_starts=A + 10 * GB, every=16, rows=4) == -3
    assert ex(flags=1, states=A + 64, cu_starts=A + 10 * GB, every=16, rows=4) == -4
    import torch
    if not torch.cuda.is_available():
        assert ex(flags=1) == -5
        assert ex(flags=0) == -5
