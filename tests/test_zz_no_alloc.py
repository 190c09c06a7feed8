"""kda_prefill_noalloc: the entry point for callers that cannot let a library
allocate device memory (an engine whose allocator owns all of HBM, a hot
path where driver allocations are forbidden).  It runs the same operation as
kda_prefill with its scratch in a fixed array inside the library.

These tests call it through the C ABI and compare it with kda_prefill on the
same inputs, and both with the FP64 oracle, within the tolerance of the other
GPU tests (per sequence and head: rel-Frobenius <= 1e-2, max-abs <= 3e-2),
over two calls in a row with different shapes, so that what the first call
leaves in the shared scratch cannot leak into the second.  This file is
collected last.
"""

import pytest
import torch

from kimi_delta_attention_kda_gb300 import _lib, build, synthetic
import kda_testutil as tu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    lib = _lib.load()
    _lib.set_split(0)
    _lib.device_status()   # clear status bits left by earlier tests
    return lib


def _ptr(t):
    return 0 if t is None else int(t.data_ptr())


def _run(raw_fn, inp):
    d = tu.to_device(inp)
    N = inp["N"]
    H = inp["q"].shape[2]
    out = torch.full_like(d["v"], float("nan"))
    fin = torch.full((N, H, 128, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    B = N if d["cu_seqlens"] is not None else inp["q"].shape[0]
    stream = torch.cuda.current_stream().cuda_stream
    rc = raw_fn(_ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]), _ptr(d["g"]), _ptr(d["beta"]),
                _ptr(d["init_state"]), _ptr(out), _ptr(fin), B, inp["q"].shape[1], H,
                _ptr(d["cu_seqlens"]), stream)
    assert rc == 0, _lib.error_string(rc)
    torch.cuda.synchronize()
    assert _lib.device_status() == 0
    return out.cpu(), fin.cpu()


def _compare(inp, got, ref):
    (o, f), (o_ref, f_ref) = got, ref
    assert torch.isfinite(o.float()).all() and torch.isfinite(f.float()).all()
    cu = inp["cu_seqlens"]
    if cu is None:
        for b in range(o.shape[0]):
            tu.assert_within_tolerance(o[b].double().numpy(), o_ref[b].double().numpy(), 1,
                                       "noalloc O seq %d" % b)
    else:
        c = cu.tolist()
        for n in range(len(c) - 1):
            if c[n + 1] > c[n]:
                tu.assert_within_tolerance(o[0, c[n]:c[n + 1]].double().numpy(),
                                           o_ref[0, c[n]:c[n + 1]].double().numpy(), 1,
                                           "noalloc O seq %d" % n)
    for n in range(f.shape[0]):
        tu.assert_within_tolerance(f[n].double().numpy(), f_ref[n].double().numpy(), 0,
                                   "noalloc final seq %d" % n)


def test_noalloc_matches_prefill_on_two_calls_in_a_row(lib):
    first = synthetic.make_inputs(0, 0, 3, 21, init_std=0.02, lengths=[40, 0, 17, 256, 1])
    second = synthetic.make_workload("t8192_h6")   # 42.5 MB of scratch: fits in 48 MiB
    got1 = _run(_lib.prefill_noalloc_raw, first)
    got2 = _run(_lib.prefill_noalloc_raw, second)
    ref1 = _run(_lib.prefill_raw, first)
    ref2 = _run(_lib.prefill_raw, second)
    _compare(first, got1, ref1)
    _compare(second, got2, ref2)
    # Both calls against the FP64 oracle as well (every head of both shapes).
    tu.check_against_oracle(first, *got1)
    tu.check_against_oracle(second, *got2)


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    """B=1, H=96, T=8192 needs about 680 MB of scratch: refused on the host
    with KDA_ERR_SCRATCH, and nothing is launched (the output stays as it was)."""
    assert _lib.noalloc_scratch_bytes() == 48 << 20
    T, H = 8192, 96
    x = torch.zeros((1, T, H, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((1, T, H, 128), dtype=torch.float32, device="cuda")
    beta = torch.zeros((1, T, H), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(x, 5.0)
    rc = _lib.prefill_noalloc_raw(_ptr(x), _ptr(x), _ptr(x), _ptr(g), _ptr(beta), 0, _ptr(out),
                                  0, 1, T, H, 0, torch.cuda.current_stream().cuda_stream)
    assert rc == -8
    assert "scratch" in _lib.error_string(rc)
    torch.cuda.synchronize()
    assert torch.all(out == 5.0)
