"""The segmented scan over chunks (kda_set_segments): each sequence cut into
segments, every segment's zero-start state and state map formed at once, a
short chain over the segments, and every segment rerun from its incoming
state.  The chunk update of "FlashKDA column split", section 1, is affine in
the incoming state (U_c is affine in S_c, and S_{c+1} = S_c D_{0:15} + U_c
K^end_c), so the results must match the FP64 oracle
within the same tolerance as the serial chain, and the serial chain itself to
rounding.  Forced segment lengths exercise ragged tails, one-segment
sequences and several sequences; the long-memory stress families check that
the incoming states really are carried across segments."""

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
    yield m
    m.set_segments(True, 0)


@pytest.fixture
def forced(kda):
    yield kda
    kda.set_segments(True, 0)


def run(kda, inp, **kw):
    d = tu.to_device(inp)
    out, fin = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                               cu_seqlens=d["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    return out.cpu(), fin.cpu()


def test_plan(kda):
    """Few heads and long sequences take the segmented scan on a GB300; a
    full head count, the packed layout, a forced split or a short sequence
    do not."""
    assert kda.plan_segments(1, 8192, 6, False) > 0
    assert kda.plan_segments(1, 65536, 1, False) > 0
    assert kda.plan_segments(1, 8192, 96, False) == 0
    assert kda.plan_segments(1, 256, 1, False) == 0
    # packed: a bound on all segments, from the total tokens
    assert kda.plan_segments(2, 16384, 6, True) > 0
    assert kda.plan_segments(8, 34816, 12, True) == 0   # 96 chains already fill most SMs
    try:
        kda.set_split(16)
        assert kda.plan_segments(1, 8192, 6, False) == 0
        kda.set_split(0)
        kda.set_segments(False)
        assert kda.plan_segments(1, 8192, 6, False) == 0
        kda.set_segments(True, 3)
        assert kda.plan_segments(1, 100, 2, False) == 3   # 7 chunks in segments of 3
    finally:
        kda.set_split(0)
        kda.set_segments(True, 0)


CASES = [(1, 256, 1, False), (2, 40, 3, True), (1, 17, 1, False), (3, 100, 2, True),
         (1, 512, 4, True), (2, 333, 2, True)]


@pytest.mark.parametrize("L", [1, 2, 3, 7])
@pytest.mark.parametrize("B,T,H,init", CASES)
def test_forced_small(forced, L, B, T, H, init):
    forced.set_segments(True, L)
    inp = synthetic.make_inputs(B, T, H, 3000 + T + L, init_std=0.02 if init else None)
    out, fin = run(forced, inp)
    tu.check_against_oracle(inp, out, fin)


@pytest.mark.parametrize("family", ["weak_decay_correlated", "model_like"])
def test_forced_long_memory(forced, family):
    """Long memory: with g = -0.01 and every key the same direction the state
    lasts for hundreds of tokens, so a wrong incoming state of any segment
    would show.  The segmented scan rounds each segment's incoming state and
    map to BF16 (relative error 2^-9 per boundary, which the serial chain's
    FP32 state does not have), so its error against the oracle may exceed
    the serial chain's by that much, not more; both stay within the
    ordinary tolerance (measured on GB300: serial 3.8e-3, segments of one
    chunk 5.4e-3 on the correlated family)."""
    import oracle
    inp = synthetic.stress_inputs(family, 1024, 2, 91)
    o_ref, f_ref = oracle.kda_token(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])
    forced.set_segments(False)
    out_s, fin_s = run(forced, inp)
    forced.set_segments(True, 5)
    out, fin = run(forced, inp)
    bound = tu.REL_FRO_TOL
    for got, ser, ref, ax in ((out[0], out_s[0], o_ref[0], 1), (fin[0], fin_s[0], f_ref[0], 0)):
        e_seg = tu.per_head_errors(got.double().numpy(), ref, ax)
        e_ser = tu.per_head_errors(ser.double().numpy(), ref, ax)
        for (rel, mx), (rel_s, _) in zip(e_seg, e_ser):
            assert rel <= bound and mx <= tu.MAX_ABS_TOL
            assert rel <= 1.15 * rel_s + 2e-3, (rel, rel_s)


def test_forced_deterministic_in_place_and_optional_states(forced):
    inp = synthetic.make_inputs(2, 300, 3, 6100, init_std=0.02)
    forced.set_segments(True, 4)
    a = run(forced, inp)
    b = run(forced, inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    d = tu.to_device(inp)
    state = d["init_state"].clone()
    out, fin = forced.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], state,
                                  final_state=state)
    torch.cuda.synchronize()
    assert forced.device_status() == 0
    assert fin.data_ptr() == state.data_ptr()
    assert torch.equal(out.cpu(), a[0]) and torch.equal(state.cpu(), a[1])
    # no initial state (zeros) and no final state requested
    inp0 = dict(inp, init_state=None)
    o0, f0 = run(forced, inp0)
    tu.check_against_oracle(inp0, o0, f0)
    d0 = tu.to_device(inp0)
    out_nf = torch.empty_like(d0["v"])
    from kimi_delta_attention_kda_gb300 import _lib
    rc = _lib.prefill_raw(d0["q"].data_ptr(), d0["k"].data_ptr(), d0["v"].data_ptr(),
                          d0["g"].data_ptr(), d0["beta"].data_ptr(), 0, out_nf.data_ptr(), 0,
                          2, 300, 3, 0, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert forced.device_status() == 0
    assert torch.equal(out_nf.cpu(), o0)


@pytest.mark.parametrize("name", ["t8192_h6", "t65536_h1"])
def test_full_workload_close_to_serial(kda, name):
    """The benchmark's plan (segmented) against the serial chain and the oracle."""
    inp = synthetic.make_workload(name)
    out, fin = run(kda, inp)
    kda.set_segments(False)
    try:
        out_s, fin_s = run(kda, inp)
    finally:
        kda.set_segments(True, 0)
    tu.assert_within_tolerance(out[0].double().numpy(), out_s[0].double().numpy(), 1,
                               "segmented vs serial O")
    tu.assert_within_tolerance(fin[0].double().numpy(), fin_s[0].double().numpy(), 0,
                               "segmented vs serial S")
    tu.check_against_oracle(inp, out, fin)


# ----------------------------------------------------------------------------
# Packed layout: segments cut on the device from cu_seqlens
# ----------------------------------------------------------------------------

LENGTHS = [40, 0, 17, 256, 1, 100]


@pytest.mark.parametrize("L", [1, 3, 7])
def test_forced_packed(forced, L):
    forced.set_segments(True, L)
    inp = synthetic.make_inputs(0, 0, 2, 7000 + L, init_std=0.02, lengths=LENGTHS)
    out, fin = run(forced, inp)
    tu.check_against_oracle(inp, out, fin)
    # empty sequence: final state = initial state
    assert torch.equal(fin[1], inp["init_state"][1])


def test_forced_packed_equals_fixed(forced):
    """Equal lengths packed and the fixed layout, cut the same way, agree bit for bit."""
    forced.set_segments(True, 5)
    inp = synthetic.make_inputs(3, 400, 2, 7100, init_std=0.02)
    out_f, fin_f = run(forced, inp)
    packed = dict(inp)
    for key in ("q", "k", "v", "g", "beta"):
        packed[key] = inp[key].reshape(1, 3 * 400, *inp[key].shape[2:]).contiguous()
    packed["cu_seqlens"] = torch.tensor([0, 400, 800, 1200], dtype=torch.int64)
    out_p, fin_p = run(forced, packed)
    assert torch.equal(out_p.reshape(out_f.shape), out_f) and torch.equal(fin_p, fin_f)


def test_forced_packed_bad_offsets_leave_outputs(forced):
    forced.set_segments(True, 2)
    H = 2
    inp = synthetic.make_inputs(1, 64, H, 7200, init_std=0.02)
    d = tu.to_device(inp)
    cu = torch.tensor([0, 40, 30, 64], dtype=torch.int64, device="cuda")
    init = torch.randn((3, H, 128, 128), device="cuda").to(torch.bfloat16)
    out = torch.full_like(d["v"], 7.0)
    fin = torch.full_like(init, 3.0)
    forced.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], init, cu_seqlens=cu, out=out,
                       final_state=fin)
    assert forced.device_status() & 1
    assert torch.all(out == 7.0) and torch.all(fin == 3.0)


def test_packed_plan_against_oracle(kda):
    """Two 8,192-token sequences at H=6: the automatic plan segments them."""
    assert kda.plan_segments(2, 16384, 6, True) > 0
    inp = synthetic.make_inputs(0, 0, 6, 7300, init_std=0.02, lengths=[8192, 6000])
    out, fin = run(kda, inp)
    kda.set_segments(False)
    try:
        out_s, fin_s = run(kda, inp)
    finally:
        kda.set_segments(True, 0)
    tu.assert_within_tolerance(out[0].double().numpy(), out_s[0].double().numpy(), 1,
                               "segmented vs serial O")
    for n in range(2):
        tu.assert_within_tolerance(fin[n].double().numpy(), fin_s[n].double().numpy(), 0,
                                   "segmented vs serial S")
    tu.check_against_oracle(inp, out, fin)


# ----------------------------------------------------------------------------
# Native checkpoints on the segmented path (the rerun writes them)
# ----------------------------------------------------------------------------

def _ck_starts(lengths, every):
    rows = [(n + every - 1) // every for n in lengths]
    out = [0]
    for r in rows:
        out.append(out[-1] + r)
    return out


def _ck_call(kda, inp, every, starts):
    d = tu.to_device(inp)
    H = inp["q"].shape[2]
    ck = torch.full((starts[-1], H, 128, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor(starts, dtype=torch.int64, device="cuda")
    out, fin, ck = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                   cu_seqlens=d["cu_seqlens"], checkpoint_every_n_tokens=every,
                                   state_checkpoints=ck, checkpoint_cu_starts=cu)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    return out.cpu(), fin.cpu(), ck.cpu()


def _check_rows(inp, lengths, every, starts, ck):
    import oracle
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    packed = inp["cu_seqlens"] is not None
    for n in range(len(lengths)):
        for j in range(starts[n + 1] - starts[n]):
            row = ck[starts[n] + j].double().numpy()
            if j == 0:
                assert torch.equal(ck[starts[n]], inp["init_state"][n])
                continue
            if packed:
                sl = slice(cu[n], cu[n] + j * every)
                args = [inp[k][:, sl] for k in ("q", "k", "v", "g", "beta")]
            else:
                args = [inp[k][n:n + 1, :j * every] for k in ("q", "k", "v", "g", "beta")]
            _, st = oracle.kda_token(*args, inp["init_state"][n:n + 1])
            tu.assert_within_tolerance(row, st[0], 0, "checkpoint seq %d row %d" % (n, j))


@pytest.mark.parametrize("every", [32, 48, 64])
def test_forced_checkpoints_fixed(forced, every):
    """Segments of 4 chunks (64 tokens); intervals of 2, 3 and 4 chunks, so
    checkpoints fall inside segments, on their boundaries and across them."""
    forced.set_segments(True, 4)
    inp = synthetic.make_inputs(2, 300, 3, 7600 + every, init_std=0.02)
    starts = _ck_starts([300, 300], every)
    out, fin, ck = _ck_call(forced, inp, every, starts)
    plain = run(forced, inp)
    assert torch.equal(out, plain[0]) and torch.equal(fin, plain[1])
    _check_rows(inp, [300, 300], every, starts, ck)
    assert forced.plan_segments(2, 300, 3, False) == 5


def test_forced_checkpoints_packed(forced):
    forced.set_segments(True, 3)
    every = 32
    inp = synthetic.make_inputs(0, 0, 2, 7700, init_std=0.02, lengths=LENGTHS)
    starts = _ck_starts(LENGTHS, every)
    out, fin, ck = _ck_call(forced, inp, every, starts)
    plain = run(forced, inp)
    assert torch.equal(out, plain[0]) and torch.equal(fin, plain[1])
    _check_rows(inp, LENGTHS, every, starts, ck)


# ----------------------------------------------------------------------------
# Two-level chain (48 or more segments per sequence, fixed layout)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("B,T,H", [(1, 1024, 1), (2, 1000, 3), (1, 800, 2), (1, 912, 2)])
def test_two_level_chain(forced, B, T, H):
    """One-chunk segments: 50-64 per sequence, composed in groups of 8 (the
    last group of 1000 tokens has 7 segments, of 800 two, of 912 one), chained
    over the groups and applied; against the oracle and the serial chain."""
    forced.set_segments(True, 1)
    assert forced.plan_segments(B, T, H, False) == (T + 15) // 16
    inp = synthetic.make_inputs(B, T, H, 7900 + T, init_std=0.02)
    out, fin = run(forced, inp)
    tu.check_against_oracle(inp, out, fin)
    forced.set_segments(False)
    out_s, fin_s = run(forced, inp)
    for b in range(B):
        tu.assert_within_tolerance(out[b].double().numpy(), out_s[b].double().numpy(), 1,
                                   "two-level vs serial O")
        tu.assert_within_tolerance(fin[b].double().numpy(), fin_s[b].double().numpy(), 0,
                                   "two-level vs serial S")


def test_two_level_chain_long_memory_and_checkpoints(forced):
    """The correlated long-memory family carries state across every group, and
    the rerun's checkpoints follow the applied incoming states."""
    import oracle
    inp = synthetic.stress_inputs("weak_decay_correlated", 1024, 2, 93)
    o_ref, f_ref = oracle.kda_token(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])
    forced.set_segments(False)
    out_s, fin_s = run(forced, inp)
    forced.set_segments(True, 1)
    out, fin = run(forced, inp)
    for got, ser, ref, ax in ((out[0], out_s[0], o_ref[0], 1), (fin[0], fin_s[0], f_ref[0], 0)):
        e_seg = tu.per_head_errors(got.double().numpy(), ref, ax)
        e_ser = tu.per_head_errors(ser.double().numpy(), ref, ax)
        for (rel, mx), (rel_s, _) in zip(e_seg, e_ser):
            assert rel <= tu.REL_FRO_TOL and mx <= tu.MAX_ABS_TOL
            assert rel <= 1.15 * rel_s + 2e-3, (rel, rel_s)
    ck_inp = synthetic.make_inputs(1, 1024, 2, 7950, init_std=0.02)
    starts = _ck_starts([1024], 128)
    o, f, ck = _ck_call(forced, ck_inp, 128, starts)
    plain = run(forced, ck_inp)
    assert torch.equal(o, plain[0]) and torch.equal(f, plain[1])
    _check_rows(ck_inp, [1024], 128, starts, ck)
