"""beta as a logit (kda_prefill_ex with KDA_FLAG_BETA_LOGIT): the operation
takes beta = sigmoid(logit) ("flashinfer kda_prefill", "Optimized Blackwell
prefill subset", beta_is_logit=True).  Checked through the C ABI against the
FP64 oracle run with the same option (per sequence and head: rel-Frobenius
<= 1e-2, max-abs <= 3e-2), on every launch plan the call can take: the
serial chain (many heads), the segmented scan (few heads, long sequence), the
one-launch form (few heads, short sequence), the packed layout with empty and
one-token sequences, and with checkpoints; plus the saturated ends, where the
mathematics fixes the answer (logit -100: beta = 0, pure decay; +100: beta = 1)."""

import math

import numpy as np
import pytest
import torch

from kimi_delta_attention_kda_gb300 import _lib, synthetic
import kda_testutil as tu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import kimi_delta_attention_kda_gb300 as m
    from kimi_delta_attention_kda_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.set_split(0)
    m.set_segments(True, 0)
    m.set_fusion(True)
    m.device_status()
    return m


def with_logits(inp, seed, std=2.0):
    """The input set with beta replaced by BF16 logits ~ N(0, std^2)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    out = dict(inp)
    out["beta"] = (std * torch.randn(inp["beta"].shape, generator=gen,
                                     dtype=torch.float32)).to(torch.bfloat16)
    return out


def run(kda, inp):
    d = tu.to_device(inp)
    out, fin = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                               cu_seqlens=d["cu_seqlens"], beta_is_logit=True)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    return out.cpu(), fin.cpu()


def check(inp, out, fin, heads=None):
    import oracle
    H = inp["q"].shape[2]
    hs = list(range(H)) if heads is None else list(heads)
    sl = lambda t: t[:, :, hs].contiguous()
    init = inp["init_state"]
    cu = inp["cu_seqlens"]
    o_ref, f_ref = oracle.kda_token(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["g"]),
                                    sl(inp["beta"]), None if init is None else init[:, hs],
                                    cu_seqlens=None if cu is None else cu.numpy(),
                                    beta_is_logit=True)
    o = out[:, :, hs].double().numpy()
    f = fin[:, hs].double().numpy()
    if cu is None:
        for b in range(o.shape[0]):
            tu.assert_within_tolerance(o[b], o_ref[b], 1, "O seq %d" % b)
    else:
        c = cu.numpy()
        for n in range(len(c) - 1):
            if c[n + 1] > c[n]:
                tu.assert_within_tolerance(o[0, c[n]:c[n + 1]], o_ref[0, c[n]:c[n + 1]], 1,
                                           "O seq %d" % n)
    for n in range(f.shape[0]):
        tu.assert_within_tolerance(f[n], f_ref[n], 0, "final seq %d" % n)


@pytest.mark.parametrize("B,T,H", [(2, 70, 3), (1, 1024, 6), (1, 8192, 6)])
def test_fixed_layout(kda, B, T, H):
    inp = with_logits(synthetic.make_inputs(B, T, H, 40 + T, init_std=0.02), 7 + T)
    out, fin = run(kda, inp)
    check(inp, out, fin)


def test_many_heads_serial_chain(kda):
    inp = with_logits(synthetic.make_inputs(1, 2048, 96, 44, init_std=0.02), 8)
    assert kda.plan_segments(1, 2048, 96, False) == 0
    out, fin = run(kda, inp)
    check(inp, out, fin, heads=[0, 47, 95])


def test_packed_with_empty_and_short_sequences(kda):
    inp = with_logits(synthetic.make_inputs(0, 0, 4, 45, init_std=0.02,
                                            lengths=[300, 0, 1, 17, 1000, 16]), 9, std=3.0)
    out, fin = run(kda, inp)
    check(inp, out, fin)


def test_matches_plain_call_on_sigmoid_of_the_logits(kda):
    """The logit path against the plain path fed BF16(sigmoid(logit)): the two
    differ only by the BF16 rounding of beta, so they agree within the
    tolerance (not bit for bit)."""
    inp = with_logits(synthetic.make_inputs(1, 512, 4, 46, init_std=0.02), 10)
    out_l, fin_l = run(kda, inp)
    d = tu.to_device(inp)
    beta = torch.sigmoid(d["beta"].float()).to(torch.bfloat16)
    out_p, fin_p = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], beta, d["init_state"])
    torch.cuda.synchronize()
    tu.assert_within_tolerance(out_l[0].double().numpy(), out_p.cpu()[0].double().numpy(), 1,
                               "logit vs plain O")
    tu.assert_within_tolerance(fin_l[0].double().numpy(), fin_p.cpu()[0].double().numpy(), 0,
                               "logit vs plain final")


def test_saturated_logits(kda):
    """logit -100: beta = 0, so the final state is S_0 with key column c scaled
    by exp(sum_t g_t[c]); logit +100: beta = 1 (checked against the oracle)."""
    T, H = 100, 2
    inp = synthetic.make_inputs(1, T, H, 47, init_std=0.3, g_low=-0.05)
    inp = dict(inp)
    inp["beta"] = torch.full((1, T, H), -100.0, dtype=torch.bfloat16)
    out, fin = run(kda, inp)
    G = inp["g"][0].double().sum(0)                                   # [H, 128]
    expect = inp["init_state"][0].double() * torch.exp(G)[:, None, :]
    tu.assert_within_tolerance(fin[0].double().numpy(), expect.numpy(), 0, "beta=0 final")
    inp["beta"] = torch.full((1, T, H), 100.0, dtype=torch.bfloat16)
    out, fin = run(kda, inp)
    check(inp, out, fin)


def test_with_checkpoints(kda):
    """Checkpoints and the logit flag together: the last row of each sequence
    equals the final state of the same call cut at that point, and O and the
    final state match the oracle."""
    T, H, every = 512, 3, 128
    inp = with_logits(synthetic.make_inputs(1, T, H, 48, init_std=0.02), 11)
    d = tu.to_device(inp)
    rows = math.ceil(T / every)
    ck = torch.zeros((rows, H, 128, 128), dtype=torch.bfloat16, device="cuda")
    cu_starts = torch.tensor([0, rows], dtype=torch.int64, device="cuda")
    out, fin, ck = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                   checkpoint_every_n_tokens=every, state_checkpoints=ck,
                                   checkpoint_cu_starts=cu_starts, beta_is_logit=True)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    check(inp, out.cpu(), fin.cpu())
    cut = {key: (val[:, :T - every].contiguous() if key in ("q", "k", "v", "g", "beta") else val)
           for key, val in inp.items()}
    _, fin_cut = run(kda, cut)
    torch.testing.assert_close(ck[rows - 1].cpu().float(), fin_cut[0].float(), rtol=2e-2, atol=2e-2)


def test_unknown_flag_is_refused(kda):
    inp = synthetic.make_inputs(1, 32, 1, 49)
    d = tu.to_device(inp)
    out = torch.empty_like(d["v"])
    rc = _lib.prefill_ex_raw(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                             d["g"].data_ptr(), d["beta"].data_ptr(), 0, out.data_ptr(), 0, 1, 32,
                             1, 0, 2, 0, 0, 0, 0, torch.cuda.current_stream().cuda_stream)
    assert rc == -7
