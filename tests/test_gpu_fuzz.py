"""Randomised shapes through the default product path, against the FP64 oracle.

A fixed list of seeds draws the layout (fixed or packed), B, T, H, the packed
lengths (empty sequences and ragged tails included) and whether there is an
initial state, so that the planner's choices (one launch, split, longest-first
order, concurrent long-sequence launch, segmented scan) meet shapes that the
hand-written cases do not.  Every (sequence, head) is held to the tolerance.
"""

import numpy as np
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


def draw(seed):
    rng = np.random.default_rng(seed)
    H = int(rng.choice([1, 2, 3, 5, 8, 12, 24, 40]))
    init = bool(rng.integers(0, 2))
    if rng.integers(0, 2):
        n = int(rng.integers(1, 9))
        lengths = [int(x) for x in rng.choice([0, 1, 15, 16, 17, 100, 333, 1024, 2500], size=n)]
        return dict(B=0, T=0, H=H, lengths=lengths, init=init)
    B = int(rng.integers(1, 4))
    T = int(rng.choice([1, 16, 31, 160, 700, 1500, 3000]))
    return dict(B=B, T=T, H=H, lengths=None, init=init)


@pytest.mark.parametrize("seed", range(24))
def test_random_shape(kda, seed):
    c = draw(1000 + seed)
    inp = synthetic.make_inputs(c["B"], c["T"], c["H"], 20000 + seed,
                                init_std=0.02 if c["init"] else None, lengths=c["lengths"])
    d = tu.to_device(inp)
    out, fin = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                               cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    tu.check_against_oracle(inp, out.cpu(), fin.cpu())
