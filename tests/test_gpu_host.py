"""kda_prefill_host: the operation on host buffers, with the host <-> device
copies overlapped with the computation.

Each case runs the host entry point on CPU tensors and checks it against the
FP64 oracle (per (sequence, head) tolerance) and against the device entry
point on the same inputs.  The cases cover each way the call cuts a batch
into pieces: token ranges of one sequence (its state handed from piece to
piece as BF16), groups of batch rows, and groups of packed sequences (with an
empty and a ragged sequence); also pageable host memory, no initial state and
no final state, zero tokens, and a CUDA-graph capture of the call.
"""

import pytest
import torch

from kimi_delta_attention_kda_gb300 import synthetic
import kda_testutil as tu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import kimi_delta_attention_kda_gb300 as m
    from kimi_delta_attention_kda_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.set_split(0)
    m.device_status()
    return m


def _pinned(inp):
    return {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _host(kda, inp, pinned=True, **kw):
    h = _pinned(inp) if pinned else inp
    out, fin = kda.kda_prefill_host(h["q"], h["k"], h["v"], h["g"], h["beta"], h["init_state"],
                                    cu_seqlens=h["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    return out, fin


def _device(kda, inp):
    d = tu.to_device(inp)
    out, fin = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                               cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    return out.cpu(), fin.cpu()


CASES = {
    # three token ranges of 1,376 tokens, the state carried in BF16
    "token_ranges": dict(B=1, T=4096, H=2, lengths=None, pieces=3),
    # three groups of one batch row each
    "batch_rows": dict(B=3, T=1024, H=4, lengths=None, pieces=3),
    # groups of whole sequences (one group only the empty one), one ragged
    "packed_groups": dict(B=0, T=0, H=3, lengths=[512, 2048, 0, 1024, 256, 4096, 48], pieces=7),
    # one piece: the copies and the call on the caller's stream
    "one_piece": dict(B=2, T=768, H=2, lengths=None, pieces=1),
}


@pytest.fixture
def pieces(kda):
    from kimi_delta_attention_kda_gb300 import _lib
    yield _lib.set_host_pieces
    _lib.set_host_pieces(0)


@pytest.mark.parametrize("case", list(CASES))
def test_host_matches_oracle_and_device(kda, pieces, case):
    c = CASES[case]
    pieces(c["pieces"])
    inp = synthetic.make_inputs(c["B"], c["T"], c["H"], 9100, init_std=0.02, lengths=c["lengths"])
    out, fin = _host(kda, inp)
    tu.check_against_oracle(inp, out, fin)
    eo, ef = _device(kda, inp)
    N = inp["init_state"].shape[0]
    tu.assert_within_tolerance(out.double().numpy().reshape(-1, c["H"], 128),
                               eo.double().numpy().reshape(-1, c["H"], 128), 1, "O host vs device")
    tu.assert_within_tolerance(fin.double().numpy().reshape(N * c["H"], 128, 128),
                               ef.double().numpy().reshape(N * c["H"], 128, 128), 0,
                               "final host vs device")


def test_host_full_workload(kda):
    """B=1, T=8192, H=6 (automatic: two token ranges) through the host path,
    against the device call (all heads) and the oracle (head 0)."""
    inp = synthetic.make_workload("t8192_h6")
    out, fin = _host(kda, inp)
    eo, ef = _device(kda, inp)
    tu.assert_within_tolerance(out[0].double().numpy(), eo[0].double().numpy(), 1, "O")
    tu.assert_within_tolerance(fin[0].double().numpy(), ef[0].double().numpy(), 0, "final")
    tu.check_against_oracle(inp, out, fin, heads=[0])


def test_host_pageable_and_no_states(kda, pieces):
    pieces(2)
    inp = synthetic.make_inputs(1, 2048, 2, 9200, init_std=None)
    pinned, _ = _host(kda, inp, output_final_state=False)
    pageable, fin = _host(kda, inp, pinned=False)
    assert torch.equal(pinned, pageable)
    tu.check_against_oracle(inp, pageable, fin)


def test_host_zero_tokens(kda):
    inp = synthetic.make_inputs(2, 0, 3, 9300, init_std=0.02)
    out, fin = _host(kda, inp)
    assert out.numel() == 0 and torch.equal(fin, inp["init_state"])


def test_host_graph_capture(kda, pieces):
    """The call (pinned buffers, three pieces) captured in a CUDA graph
    replays what an eager call computes, bit for bit, on fresh inputs."""
    pieces(3)
    first = _pinned(synthetic.make_inputs(1, 4096, 2, 9400, init_std=0.02))
    second = synthetic.make_inputs(1, 4096, 2, 9500, init_std=0.02)
    static = {k: (v.clone().pin_memory() if isinstance(v, torch.Tensor) else v)
              for k, v in first.items()}
    out = torch.empty(static["v"].shape, dtype=torch.bfloat16).pin_memory()
    fin = torch.empty(static["init_state"].shape, dtype=torch.bfloat16).pin_memory()

    def call():
        kda.kda_prefill_host(static["q"], static["k"], static["v"], static["g"], static["beta"],
                             static["init_state"], out=out, final_state=fin)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    torch.cuda.synchronize()
    for inp in (second, first):
        for key, v in inp.items():
            if isinstance(v, torch.Tensor):
                static[key].copy_(v)
        graph.replay()
        torch.cuda.synchronize()
        assert kda.device_status() == 0
        got = (out.clone(), fin.clone())
        eo, ef = _host(kda, inp)
        assert torch.equal(got[0], eo) and torch.equal(got[1], ef)


def test_launch_counts(kda):
    """kda_last_call_launches reports the kernels one call enqueued: the
    preparation and the recurrence (more heads than SMs); one cooperative
    launch (many heads, or few heads and a short sequence); the segmented
    scan's four kernels (six with the two-level chain); a packed batch in the
    many-head form: the offsets' metadata, the chunk order and one
    cooperative launch."""
    from kimi_delta_attention_kda_gb300 import _lib
    for (B, T, H), want in (((2, 2048, 96), 2), ((1, 2048, 96), 1), ((1, 256, 1), 1),
                            ((1, 8192, 6), 4), ((1, 65536, 1), 6)):
        d = tu.to_device(synthetic.make_inputs(B, T, H, 9600, init_std=0.02))
        kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"])
        torch.cuda.synchronize()
        assert _lib.last_call_launches() == want, (B, T, H)
    d = tu.to_device(synthetic.make_workload("varlen8_h12"))
    kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                    cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert _lib.last_call_launches() == 3
