"""GPU parity on the degenerate and boundary cases of the method, against
the FP64 oracle (and, where the mathematics fixes the answer, a closed form).

- beta = 0: no write ever happens, so the state only decays:
  S_T = S_0 Diag(exp(sum_t g_t)) (column-wise), o_t = s S_0 Diag(exp(G_t)) qhat_t.
- g = 0: no decay (the plain delta rule).
- More (sequence, head) chains than SMs in a fixed-length batch (several
  waves of recurrence CTAs), and many heads on few tokens.
- A packed batch whose sequences are each shorter than one chunk.
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


def run(kda, inp):
    d = tu.to_device(inp)
    out, fin = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                               cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    return out.cpu(), fin.cpu()


@pytest.mark.parametrize("T", [16, 300, 2048])
def test_beta_zero_is_pure_decay(kda, T):
    inp = synthetic.make_inputs(1, T, 3, 9700 + T, init_std=0.5)
    inp["beta"] = torch.zeros_like(inp["beta"])
    out, fin = run(kda, inp)
    tu.check_against_oracle(inp, out, fin)
    # Closed form of the final state: every key column of S_0 scaled by
    # exp(sum of its log-decays).
    S0 = inp["init_state"].double().numpy()[0]                     # [H, V, K]
    gsum = inp["g"].double().numpy()[0].sum(axis=0)                 # [H, K]
    ref = S0 * np.exp(gsum)[:, None, :]
    got = fin.double().numpy()[0]
    for h in range(ref.shape[0]):
        den = np.linalg.norm(ref[h])
        assert np.linalg.norm(got[h] - ref[h]) <= 1e-2 * den + 1e-6
        assert np.abs(got[h] - ref[h]).max() <= 3e-2


@pytest.mark.parametrize("T", [40, 1024])
def test_no_decay(kda, T):
    inp = synthetic.make_inputs(2, T, 2, 9800 + T, init_std=0.02)
    inp["g"] = torch.zeros_like(inp["g"])
    out, fin = run(kda, inp)
    tu.check_against_oracle(inp, out, fin)


def test_multi_wave_fixed_batch(kda):
    """3 x 64 = 192 (sequence, head) chains on 152 SMs."""
    inp = synthetic.make_inputs(3, 80, 64, 9900, init_std=0.02)
    out, fin = run(kda, inp)
    tu.check_against_oracle(inp, out, fin)


@pytest.mark.parametrize("B,T,H", [(1, 33, 160), (2, 48, 512)])
def test_many_heads_few_tokens(kda, B, T, H):
    """Recurrence grids of several waves (up to 1,024 CTAs) and preparation
    grids with more items than pairs."""
    inp = synthetic.make_inputs(B, T, H, 9910 + H, init_std=0.02)
    out, fin = run(kda, inp)
    tu.check_against_oracle(inp, out, fin)


def test_packed_sub_chunk_sequences(kda):
    inp = synthetic.make_inputs(0, 0, 4, 9920, init_std=0.02,
                                lengths=[1, 15, 7, 0, 3, 16, 9, 2, 11, 5])
    out, fin = run(kda, inp)
    tu.check_against_oracle(inp, out, fin)


@pytest.mark.parametrize("T", [16, 500])
def test_read_back_closed_form(kda, T):
    """No decay (g = 0), beta = 1 and q = k: after token t's write
    S khat_t = v_t exactly (khat has unit norm), so o_t = s v_t whatever the
    initial state: a closed form that needs no oracle."""
    inp = synthetic.make_inputs(1, T, 2, 9930 + T, init_std=0.5)
    inp["q"] = inp["k"].clone()
    inp["g"] = torch.zeros_like(inp["g"])
    inp["beta"] = torch.ones_like(inp["beta"])
    out, fin = run(kda, inp)
    ref = inp["v"].double().numpy()[0] / np.sqrt(128.0)             # [T, H, 128]
    got = out.double().numpy()[0]
    tu.assert_within_tolerance(got, ref, 1, "O against s v")
    tu.check_against_oracle(inp, out, fin)
