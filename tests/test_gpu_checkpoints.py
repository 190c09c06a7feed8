"""Native state checkpoints ("flashinfer kda_prefill", Native checkpoints):
kda_prefill_checkpointed writes the state before every interval of each
sequence.  A checkpoint is the recurrence's own state at a chunk boundary, so
row j of a sequence must equal, bit for bit, the final state of the same call
cut after j intervals (same kernel variant); packed sequences are also checked
against the oracle."""

import numpy as np
import pytest
import torch

import oracle
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
    # Checkpointed calls always run the serial chain; the plain calls they are
    # compared with bit for bit must too.
    m.set_segments(False)
    m.device_status()
    yield m
    m.set_split(0)
    m.set_engine(0)
    m.set_segments(True)


def _rows(lengths, every):
    return [(n + every - 1) // every for n in lengths]


def _starts(lengths, every):
    return [0] + list(np.cumsum(_rows(lengths, every)))


def _call(kda, inp, every, starts, rows=None, fill=0.0):
    d = tu.to_device(inp)
    H = inp["q"].shape[2]
    rows = starts[-1] if rows is None else rows
    ck = torch.full((rows, H, 128, 128), fill, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor(starts, dtype=torch.int64, device="cuda")
    out, fin, ck = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                   cu_seqlens=d["cu_seqlens"], checkpoint_every_n_tokens=every,
                                   state_checkpoints=ck, checkpoint_cu_starts=cu)
    torch.cuda.synchronize()
    return out.cpu(), fin.cpu(), ck.cpu()


def _plain(kda, inp):
    d = tu.to_device(inp)
    out, fin = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                               cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    return out.cpu(), fin.cpu()


def _prefix(inp, T):
    """The fixed-layout input cut after T tokens."""
    p = dict(inp)
    for key in ("q", "k", "v", "g", "beta"):
        p[key] = inp[key][:, :T].contiguous()
    return p


def _check_against_prefixes(kda, inp, every):
    B, T, H = inp["q"].shape[:3]
    starts = _starts([T] * B, every)
    out, fin, ck = _call(kda, inp, every, starts)
    assert kda.device_status() == 0
    ref_out, ref_fin = _plain(kda, inp)
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)   # checkpoints change nothing else
    init = inp["init_state"] if inp["init_state"] is not None else torch.zeros(B, H, 128, 128,
                                                                              dtype=torch.bfloat16)
    for b in range(B):
        assert torch.equal(ck[starts[b]], init[b])
        for j in range(1, starts[b + 1] - starts[b]):
            _, pf = _plain(kda, _prefix(inp, j * every))
            assert torch.equal(ck[starts[b] + j], pf[b]), (b, j)


@pytest.mark.parametrize("engine,nsplit", [(0, 0), (0, 1), (0, 2), (0, 4), (0, 8), (0, 16),
                                           (1, 4), (1, 8)])
def test_checkpoints_equal_prefix_states(kda, engine, nsplit):
    """Every recurrence variant: 4 x 32 columns (split 1), 8 x 8 (split 2),
    key split (4, 8, 16; one launch with the preparation at 8 and 16 here),
    and the keys-major warps of engine 1."""
    kda.set_split(nsplit)
    kda.set_engine(engine)
    try:
        _check_against_prefixes(kda, synthetic.make_inputs(2, 300, 3, 5100, init_std=0.02), 64)
    finally:
        kda.set_split(0)
        kda.set_engine(0)


def test_checkpoints_one_cta_per_head_and_one_launch(kda):
    """B=1, T=8192 at H=96 (4 warps x 32 columns: a call with checkpoints runs
    the two kernels) and at H=6 (preparation and recurrence in one launch)."""
    assert kda.plan_fused(1, 8192, 6, False)
    for name, every in (("t8192_h96", 2048), ("t8192_h6", 1024)):
        _check_against_prefixes(kda, synthetic.make_workload(name), every)


def test_checkpoints_packed_against_oracle(kda):
    lengths = [40, 0, 17, 256, 1, 100]
    every = 32
    inp = synthetic.make_inputs(0, 0, 3, 5200, init_std=0.02, lengths=lengths)
    starts = _starts(lengths, every)
    out, fin, ck = _call(kda, inp, every, starts)
    assert kda.device_status() == 0
    ref_out, ref_fin = _plain(kda, inp)
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    cu = inp["cu_seqlens"].tolist()
    for n, L in enumerate(lengths):
        for j in range(starts[n + 1] - starts[n]):
            t0, t1 = cu[n], cu[n] + j * every
            if j == 0:
                ref = inp["init_state"][n].double().numpy()
            else:
                sl = slice(t0, t1)
                _, st = oracle.kda_token(inp["q"][:, sl], inp["k"][:, sl], inp["v"][:, sl],
                                         inp["g"][:, sl], inp["beta"][:, sl],
                                         inp["init_state"][n:n + 1])
                ref = st[0]
            tu.assert_within_tolerance(ck[starts[n] + j].double().numpy(), ref, 0,
                                       "checkpoint seq %d row %d" % (n, j))


def test_bad_offsets_are_reported_and_skipped(kda):
    """Offsets that give a sequence fewer rows than it has checkpoints: the
    missing ones are not written (no row outside the sequence's range or the
    buffer is touched) and KDA_DEV_BAD_CHECKPOINTS is set."""
    inp = synthetic.make_inputs(2, 300, 2, 5300, init_std=0.02)   # 5 checkpoints per sequence
    starts = [0, 3, 6]                                              # room for 3 each
    sentinel = 7.0
    out, fin, ck = _call(kda, inp, 64, starts, rows=8, fill=sentinel)
    assert kda.device_status() == 4
    full_out, full_fin, full_ck = _call(kda, inp, 64, _starts([300, 300], 64))
    assert kda.device_status() == 0
    assert torch.equal(out, full_out) and torch.equal(fin, full_fin)
    assert torch.equal(ck[0:3], full_ck[0:3])      # sequence 0, rows 0-2
    assert torch.equal(ck[3:6], full_ck[5:8])      # sequence 1, rows 0-2
    assert torch.all(ck[6:8] == sentinel)          # never written


def test_engine2_calls_with_checkpoints_use_the_column_split(kda):
    inp = synthetic.make_inputs(1, 160, 2, 5400, init_std=0.02)
    a = _call(kda, inp, 32, _starts([160], 32))
    kda.set_engine(2)
    try:
        b = _call(kda, inp, 32, _starts([160], 32))
    finally:
        kda.set_engine(0)
    assert kda.device_status() == 0
    for x, y in zip(a, b):
        assert torch.equal(x, y)
