"""The bounded waits' exit path, on the GPU, without a fault or a hang.

Every wait in the library's kernels (mbarrier waits of the TMA rings, the
ready-flag poll of the one-launch form) gives up after a bound (about 2 s in
libkda.so), sets KDA_DEV_PIPE_TIMEOUT and returns.  The test library
libkda_testhooks.so compiles the same waits with a bound of 10^5 cycles and
runs them where they cannot complete: a ring whose fourth stage no producer
fills, and a ready flag that nothing sets.  Each wait must run out, set the
status bit and return; then the GPU must still answer: a normal kda_prefill
on the same device matches the oracle."""

import ctypes

import pytest
import torch

from kimi_delta_attention_kda_gb300 import build, synthetic
import kda_testutil as tu

pytestmark = pytest.mark.gpu

KDA_DEV_PIPE_TIMEOUT = 2


@pytest.fixture(scope="module")
def hooks():
    build.build()
    path = build.build_test_hooks()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.kda_test_wait_bounds.argtypes = [P, P, P, P, P]
    lib.kda_test_wait_bounds.restype = ctypes.c_int
    lib.kda_test_wait_bound_cycles.argtypes = []
    lib.kda_test_wait_bound_cycles.restype = ctypes.c_longlong
    return lib


def test_waits_run_out_and_report(hooks):
    assert hooks.kda_test_wait_bound_cycles() == build.TEST_WAIT_BOUND_CYCLES
    src = torch.arange(4096, dtype=torch.int32, device="cuda").to(torch.uint8)
    flags = torch.zeros(32, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    rc = hooks.kda_test_wait_bounds(src.data_ptr(), flags.data_ptr(), status.data_ptr(),
                                    out.data_ptr(), stream.cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()            # returns: no wait hung
    seen, ring_timed_out, flag_timed_out = out.tolist()
    assert seen == 3                    # the three filled stages were consumed
    assert ring_timed_out == 1          # the unfilled fourth stage ran out
    assert flag_timed_out == 1          # the flag nobody sets ran out
    assert int(status.item()) & KDA_DEV_PIPE_TIMEOUT


def test_gpu_still_answers(hooks):
    """After the timeouts the context is intact: a normal call is correct."""
    import kimi_delta_attention_kda_gb300 as kda
    kda.device_status()
    inp = synthetic.make_inputs(1, 100, 2, 5, init_std=0.02)
    d = tu.to_device(inp)
    out, fin = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"])
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    tu.check_against_oracle(inp, out.cpu(), fin.cpu())
