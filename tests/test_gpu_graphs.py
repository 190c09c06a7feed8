"""kda_prefill under CUDA-graph capture.

The call is stream-ordered with no host synchronisation and no host read of
device data ("flashinfer kda_prefill", State and graph semantics), and its
workspace comes from a stream-ordered pool, so it can be captured into a CUDA
graph and replayed.  Each launch form is captured once and replayed on fresh
inputs; replays must equal eager calls bit for bit: the segmented scan (fixed
and packed), the one cooperative launch, the packed batch with its concurrent
second launch on the library's side stream, and one CTA per head.
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


CASES = {
    "segmented_fixed": dict(B=1, T=8192, H=6, lengths=None),
    "one_launch": dict(B=1, T=1024, H=6, lengths=None),
    # mean below 64 chunks: the two-kernel path, the longest four at split 2
    "packed_long_split": dict(B=0, T=0, H=12, lengths=[3072, 256, 512, 1024, 128, 1536, 384, 768]),
    # the many-head one-launch form (metadata, chunk order, one cooperative launch)
    "packed_one_launch": dict(B=0, T=0, H=12, lengths=[4096, 512, 1024, 2048, 256, 3072, 768, 1536]),
    "segmented_packed": dict(B=0, T=0, H=6, lengths=[8192, 6000]),
    "one_cta_per_head": dict(B=1, T=2048, H=96, lengths=None),
}


def _inputs(case, seed):
    c = CASES[case]
    return synthetic.make_inputs(c["B"], c["T"], c["H"], seed, init_std=0.02, lengths=c["lengths"])


@pytest.mark.parametrize("case", list(CASES))
def test_graph_replay_equals_eager(kda, case):
    first = tu.to_device(_inputs(case, 8100))
    second = tu.to_device(_inputs(case, 8200))
    H = first["q"].shape[2]
    N = first["init_state"].shape[0]
    if case.startswith("packed"):
        T = first["q"].shape[1]
        assert kda.plan_fused(N, T, H, True) == (case == "packed_one_launch")
        assert (kda.plan_long_split(N, T, H) > 0) == (case == "packed_long_split")
    # Static buffers the graph reads and writes.
    static = {k: (None if v is None else v.clone()) for k, v in first.items()}
    out = torch.empty_like(static["v"])
    fin = torch.empty((N, H, 128, 128), dtype=torch.bfloat16, device="cuda")

    def call():
        kda.kda_prefill(static["q"], static["k"], static["v"], static["g"], static["beta"],
                        static["init_state"], cu_seqlens=static["cu_seqlens"], out=out,
                        final_state=fin)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()                      # warm-up outside the capture (library state, pool)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    torch.cuda.synchronize()
    assert kda.device_status() == 0

    for inp in (first, second, first):
        for key, v in inp.items():
            if v is not None:
                static[key].copy_(v)
        graph.replay()
        torch.cuda.synchronize()
        assert kda.device_status() == 0
        got = (out.clone(), fin.clone())
        eo, ef = kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                 inp["init_state"], cu_seqlens=inp["cu_seqlens"])
        torch.cuda.synchronize()
        assert torch.equal(got[0], eo) and torch.equal(got[1], ef), case
