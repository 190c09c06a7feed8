"""Pins of the FP64 oracle to facts that do not come from the oracle itself.

Every test here runs on the CPU.  The pins are chosen so that a plausible
mistake in the oracle (a dropped term, a wrong sign, a decay applied to the
wrong side of the state, an off-by-one in the decay products, a transposed
operand) fails at least one of them:

* hand-computed recurrences (``golden/hand_recurrence.json``);
* closed forms: pure decay (beta = 0), exact read-back (alpha = 1, beta = 1,
  q = k), orthonormal keys;
* structure: linearity in (V, S_0), channel permutations, scale invariance of
  the normalised q and k, packed = separate, split-and-continue, the affine
  segment maps S -> S F + Z and their composition;
* the second, chunkwise implementation (no shared code) for several chunk
  lengths and both inverse methods;
* (I + R)^{-1} against a library inverse and its defining residual;
* the split-exponent form of the chunk quantities against the product form.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from kimi_delta_attention_kda_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def small_inputs(B=2, T=37, H=2, d=16, seed=0, init=True, **kw):
    return synthetic.make_inputs(B, T, H, seed, dk=d, dv=d,
                                 init_std=0.5 if init else None, **kw)


def f64(x):
    return None if x is None else x.double().numpy()


# --------------------------------------------------------------------------
# Hand-computed cases
# --------------------------------------------------------------------------

def _hand_cases():
    with open(os.path.join(GOLDEN, "hand_recurrence.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _hand_cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("form", ["token", "chunk1", "chunk2", "chunk3", "chunk16"])
def test_hand_computed(oracle_mod, case, form):
    dk, dv = case["dk"], case["dv"]
    T = len(case["beta"])
    q = np.array(case["q"], dtype=np.float64).reshape(1, T, 1, dk)
    k = np.array(case["k"], dtype=np.float64).reshape(1, T, 1, dk)
    v = np.array(case["v"], dtype=np.float64).reshape(1, T, 1, dv)
    g = np.log(np.array(case["alpha"], dtype=np.float64)).reshape(1, T, 1, dk)
    beta = np.array(case["beta"], dtype=np.float64).reshape(1, T, 1)
    init = None
    if case["init"] is not None:
        init = np.array(case["init"], dtype=np.float64).reshape(1, 1, dv, dk)
    if form == "token":
        out, fin = oracle_mod.kda_token(q, k, v, g, beta, init, scale=case["scale"], eps=0.0)
    else:
        C = int(form[len("chunk"):])
        out, fin = oracle_mod.kda_chunk(q, k, v, g, beta, init, scale=case["scale"], eps=0.0,
                                        chunk=C)
    np.testing.assert_allclose(out.reshape(T, dv), np.array(case["out"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(fin.reshape(dv, dk), np.array(case["final"]), rtol=0,
                               atol=1e-14)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

def _normalise(x, eps=1e-6):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


def test_beta_zero_is_pure_decay(oracle_mod):
    """beta = 0: nothing is written, so S_t = S_0 Diag(exp(G_t)) with G_t the
    running sum of g over the sequence, and o_t = s S_t qhat_t."""
    inp = small_inputs(B=1, T=29, H=1, d=8, seed=3)
    q, k, v, g = map(f64, (inp["q"], inp["k"], inp["v"], inp["g"]))
    S0 = f64(inp["init_state"])[0, 0]
    beta = np.zeros((1, 29, 1))
    out, fin = oracle_mod.kda_token(q, k, v, g, beta, S0[None, None])
    G = np.cumsum(g[0, :, 0, :], axis=0)          # [T, dk]
    qh = _normalise(q[0, :, 0, :])
    s = 1 / math.sqrt(8)
    expect = np.stack([s * (S0 * np.exp(G[t])[None, :]) @ qh[t] for t in range(29)])
    assert rel_fro(out[0, :, 0, :], expect) < 1e-13
    assert rel_fro(fin[0, 0], S0 * np.exp(G[-1])[None, :]) < 1e-13
    # The value input must not matter at all.
    out2, _ = oracle_mod.kda_token(q, k, 100 * v + 3, g, beta, S0[None, None])
    np.testing.assert_array_equal(out, out2)


def test_exact_readback(oracle_mod):
    """alpha = 1, beta = 1 and q = k: the write makes S_t khat_t = v_t exactly,
    so o_t = s v_t whatever came before (||khat|| = 1 with eps = 0)."""
    inp = small_inputs(B=1, T=40, H=3, d=16, seed=5)
    k, v = f64(inp["k"]), f64(inp["v"])
    g = np.zeros_like(k)
    beta = np.ones(k.shape[:3])
    out, _ = oracle_mod.kda_token(k, k, v, g, beta, f64(inp["init_state"]), eps=0.0)
    np.testing.assert_allclose(out, v / 4.0, rtol=0, atol=1e-12)


def test_orthonormal_keys_closed_form(oracle_mod):
    """alpha = 1, beta = 1, orthonormal keys: S_T = S_0 + sum_t (v_t - S_0 k_t) k_t^T."""
    d, T = 16, 12
    rng = np.random.default_rng(7)
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    keys = Qm[:, :T].T                       # T orthonormal rows
    v = rng.standard_normal((T, d))
    S0 = rng.standard_normal((d, d))
    q = rng.standard_normal((T, d))
    out, fin = oracle_mod.kda_token(q.reshape(1, T, 1, d), keys.reshape(1, T, 1, d),
                                    v.reshape(1, T, 1, d), np.zeros((1, T, 1, d)),
                                    np.ones((1, T, 1)), S0.reshape(1, 1, d, d), eps=0.0)
    expect = S0 + sum(np.outer(v[t] - S0 @ keys[t], keys[t]) for t in range(T))
    assert rel_fro(fin[0, 0], expect) < 1e-13


# --------------------------------------------------------------------------
# Structure
# --------------------------------------------------------------------------

def test_linear_in_values_and_state(oracle_mod):
    """For fixed q, k, g, beta the map (V, S_0) -> (O, S_T) is linear."""
    a = small_inputs(B=1, T=33, H=2, d=16, seed=11)
    b = small_inputs(B=1, T=33, H=2, d=16, seed=12)
    q, k, g, beta = map(f64, (a["q"], a["k"], a["g"], a["beta"]))
    v1, v2 = f64(a["v"]), f64(b["v"])
    s1, s2 = f64(a["init_state"]), f64(b["init_state"])
    o1, f1 = oracle_mod.kda_token(q, k, v1, g, beta, s1)
    o2, f2 = oracle_mod.kda_token(q, k, v2, g, beta, s2)
    o3, f3 = oracle_mod.kda_token(q, k, 2.5 * v1 - 0.5 * v2, g, beta, 2.5 * s1 - 0.5 * s2)
    assert rel_fro(o3, 2.5 * o1 - 0.5 * o2) < 1e-12
    assert rel_fro(f3, 2.5 * f1 - 0.5 * f2) < 1e-12


def test_channel_permutations(oracle_mod):
    """Permuting key channels (q, k, g and the state's columns together) leaves
    O unchanged and permutes the final state's columns; permuting value
    channels permutes O and the state's rows.  Catches a transposed state."""
    inp = small_inputs(B=1, T=31, H=1, d=16, seed=21)
    q, k, v, g, beta, s0 = map(f64, (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["init_state"]))
    o, f = oracle_mod.kda_token(q, k, v, g, beta, s0)
    rng = np.random.default_rng(0)
    pk = rng.permutation(16)
    pv = rng.permutation(16)
    o_k, f_k = oracle_mod.kda_token(q[..., pk], k[..., pk], v, g[..., pk], beta, s0[..., pk])
    assert rel_fro(o_k, o) < 1e-13
    assert rel_fro(f_k, f[..., pk]) < 1e-13
    o_v, f_v = oracle_mod.kda_token(q, k, v[..., pv], g, beta, s0[:, :, pv, :])
    assert rel_fro(o_v, o[..., pv]) < 1e-13
    assert rel_fro(f_v, f[:, :, pv, :]) < 1e-13


def test_qk_scale_invariance(oracle_mod):
    """q and k are normalised in the operation: positive rescaling of either
    changes nothing (with eps = 0)."""
    inp = small_inputs(B=1, T=20, H=2, d=16, seed=4)
    q, k, v, g, beta, s0 = map(f64, (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["init_state"]))
    o, f = oracle_mod.kda_token(q, k, v, g, beta, s0, eps=0.0)
    scale_q = np.exp(np.random.default_rng(1).uniform(-3, 3, size=q.shape[:3] + (1,)))
    o2, f2 = oracle_mod.kda_token(q * scale_q, k * 7.0, v, g, beta, s0, eps=0.0)
    assert rel_fro(o2, o) < 1e-13 and rel_fro(f2, f) < 1e-13


@pytest.mark.parametrize("form", ["token", "chunk"])
def test_packed_equals_separate(oracle_mod, form):
    """Packed sequences never interact: each one equals its own run."""
    lengths = [5, 0, 33, 16, 1]
    inp = synthetic.make_inputs(0, 0, 2, 9, dk=16, dv=16, init_std=0.3, lengths=lengths)
    q, k, v, g, beta, s0 = map(f64, (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["init_state"]))
    cu = inp["cu_seqlens"].numpy()
    fn = oracle_mod.kda_token if form == "token" else oracle_mod.kda_chunk
    out, fin = fn(q, k, v, g, beta, s0, cu_seqlens=cu)
    for n, L in enumerate(lengths):
        a, b = cu[n], cu[n + 1]
        if L == 0:
            np.testing.assert_array_equal(fin[n], s0[n])
            continue
        o1, f1 = fn(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], s0[n:n + 1])
        np.testing.assert_allclose(out[:, a:b], o1, rtol=0, atol=1e-15)
        np.testing.assert_allclose(fin[n], f1[0], rtol=0, atol=1e-15)


def test_split_and_continue(oracle_mod):
    """Running tokens [0, t0) then [t0, T) from the carried state equals one run."""
    inp = small_inputs(B=1, T=45, H=2, d=16, seed=8)
    q, k, v, g, beta, s0 = map(f64, (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["init_state"]))
    o, f = oracle_mod.kda_token(q, k, v, g, beta, s0)
    for t0 in (1, 16, 23):
        oa, fa = oracle_mod.kda_token(q[:, :t0], k[:, :t0], v[:, :t0], g[:, :t0],
                                      beta[:, :t0], s0)
        ob, fb = oracle_mod.kda_chunk(q[:, t0:], k[:, t0:], v[:, t0:], g[:, t0:],
                                      beta[:, t0:], fa)
        assert rel_fro(np.concatenate([oa, ob], axis=1), o) < 1e-12
        assert rel_fro(fb, f) < 1e-12


def test_segment_maps_compose(oracle_mod):
    """With the keys, decays and betas fixed, a run of tokens maps the state
    affinely, S_end = S_0 F + Z: F is the end state from S_0 = I with V = 0
    (each value row evolves on its own, S <- S Diag(alpha)(I - beta k k^T)),
    Z the end state from zero.  Consecutive runs compose, (F1, Z1) then
    (F2, Z2) = (F1 F2, Z1 F2 + Z2), which is what a scan over segments of
    chunks, and over groups of segments, relies on."""
    d, H = 16, 2
    # Weak decay, so that F keeps the incoming state (with g down to -5 it
    # would be close to zero after a few tokens and pin nothing).
    inp = small_inputs(B=1, T=48, H=H, d=d, seed=13, g_low=-0.05)
    q, k, v, g, beta, s0 = map(f64, (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["init_state"]))
    eye = np.broadcast_to(np.eye(d), (1, H, d, d)).copy()
    cuts = [0, 7, 23, 30, 48]
    maps = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = (q[:, a:b], k[:, a:b])
        _, f = oracle_mod.kda_token(*part, np.zeros_like(v[:, a:b]), g[:, a:b], beta[:, a:b], eye)
        _, z = oracle_mod.kda_token(*part, v[:, a:b], g[:, a:b], beta[:, a:b], None)
        maps.append((f, z))
    _, ref = oracle_mod.kda_token(q, k, v, g, beta, s0)
    s = s0
    for f, z in maps:
        s = s @ f + z
    assert rel_fro(s, ref) < 1e-12
    # The first two segments' maps composed into one, then the rest.
    (f1, z1), (f2, z2) = maps[0], maps[1]
    s = s0 @ (f1 @ f2) + (z1 @ f2 + z2)
    for f, z in maps[2:]:
        s = s @ f + z
    assert rel_fro(s, ref) < 1e-12
    # Planted mistakes are caught: the map applied from the left, or transposed.
    for wrong in (lambda s, f: f @ s, lambda s, f: s @ np.swapaxes(f, -1, -2)):
        s = s0
        for f, z in maps:
            s = wrong(s, f) + z
        assert rel_fro(s, ref) > 1e-2


def test_empty_sequences(oracle_mod):
    """T = 0: the final state is the initial state and nothing is written."""
    inp = small_inputs(B=3, T=0, H=2, d=8, seed=1)
    q, k, v, g, beta, s0 = map(f64, (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["init_state"]))
    out, fin = oracle_mod.kda_token(q, k, v, g, beta, s0)
    assert out.size == 0
    np.testing.assert_array_equal(fin, s0)
    _, fin2 = oracle_mod.kda_chunk(q, k, v, g, beta, s0)
    np.testing.assert_array_equal(fin2, s0)


def test_zero_key_writes_nothing(oracle_mod):
    """A zero key normalises to zero (the eps keeps it finite), so its token
    only decays the state and leaves it otherwise untouched."""
    inp = small_inputs(B=1, T=3, H=1, d=8, seed=2)
    q, k, v, g, beta, s0 = map(f64, (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["init_state"]))
    k[0, 1] = 0.0
    o, f = oracle_mod.kda_token(q[:, :2], k[:, :2], v[:, :2], g[:, :2], beta[:, :2], s0)
    o1, f1 = oracle_mod.kda_token(q[:, :1], k[:, :1], v[:, :1], g[:, :1], beta[:, :1], s0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(f))
    assert rel_fro(f, f1 * np.exp(g[0, 1, 0])[None, None, None, :]) < 1e-14


# --------------------------------------------------------------------------
# Second implementation: the chunkwise form
# --------------------------------------------------------------------------

@pytest.mark.parametrize("chunk", [1, 3, 8, 16, 32])
@pytest.mark.parametrize("inverse", ["forward", "neumann"])
def test_chunkwise_matches_token(oracle_mod, chunk, inverse):
    inp = small_inputs(B=2, T=53, H=2, d=32, seed=100 + chunk)
    args = [inp[n] for n in ("q", "k", "v", "g", "beta", "init_state")]
    o_t, f_t = oracle_mod.kda_token(*args)
    o_c, f_c = oracle_mod.kda_chunk(*args, chunk=chunk, inverse=inverse)
    assert rel_fro(o_c, o_t) < 1e-10
    assert rel_fro(f_c, f_t) < 1e-10


def test_chunkwise_matches_token_head_dim_128(oracle_mod):
    inp = synthetic.make_inputs(1, 70, 2, 17, init_std=0.02)
    args = [inp[n] for n in ("q", "k", "v", "g", "beta", "init_state")]
    o_t, f_t = oracle_mod.kda_token(*args)
    o_c, f_c = oracle_mod.kda_chunk(*args, chunk=16)
    assert rel_fro(o_c, o_t) < 1e-10
    assert rel_fro(f_c, f_t) < 1e-10


@pytest.mark.parametrize("family", ["floor_e-5", "weak_decay_correlated", "model_like"])
def test_chunkwise_matches_token_stress(oracle_mod, family):
    inp = synthetic.stress_inputs(family, 64, 2, 3, dk=32, dv=32)
    args = [inp[n] for n in ("q", "k", "v", "g", "beta")]
    o_t, f_t = oracle_mod.kda_token(*args)
    for inverse in ("forward", "neumann"):
        o_c, f_c = oracle_mod.kda_chunk(*args, chunk=16, inverse=inverse)
        assert rel_fro(o_c, o_t) < 1e-10
        assert rel_fro(f_c, f_t) < 1e-10


# --------------------------------------------------------------------------
# The 16 x 16 inverse
# --------------------------------------------------------------------------

@pytest.mark.parametrize("C", [1, 2, 5, 16, 17, 32])
def test_unitri_inverse(oracle_mod, C):
    rng = np.random.default_rng(C)
    L = np.tril(rng.standard_normal((C, C)) * 0.3, -1)
    I = np.eye(C)
    Xf = oracle_mod.unitri_inverse(L, "forward")
    Xn = oracle_mod.unitri_inverse(L, "neumann")
    np.testing.assert_allclose(Xf, np.linalg.inv(I + L), rtol=0, atol=1e-12)
    assert np.abs((I + L) @ Xf - I).max() < 1e-12
    np.testing.assert_allclose(Xn, Xf, rtol=0, atol=1e-12)
    # lower unitriangular
    np.testing.assert_array_equal(np.triu(Xf, 1), 0.0)
    np.testing.assert_allclose(np.diag(Xf), 1.0, rtol=0, atol=0)


@pytest.mark.parametrize("family", ["floor_e-5", "weak_decay_correlated", "model_like"])
def test_akk_residual_stress(oracle_mod, family):
    """(I + R) A^kk = I for the chunk quantities of the stress families."""
    inp = synthetic.stress_inputs(family, 48, 2, 5, dk=128, dv=128)
    im = oracle_mod.chunk_intermediates(inp["q"], inp["k"], inp["g"], inp["beta"], chunk=16)
    kh = _normalise(f64(inp["k"])[0])                            # [T, H, dk]
    g = f64(inp["g"])[0]
    beta = f64(inp["beta"])[0]
    for ch in range(im["Akk"].shape[0]):
        for h in range(im["Akk"].shape[1]):
            sl = slice(16 * ch, 16 * ch + 16)
            G = np.cumsum(g[sl, h], axis=0)
            R = np.zeros((16, 16))
            for i in range(16):
                for j in range(i):
                    R[i, j] = beta[sl][i, h] * np.sum(kh[sl][j, h] * kh[sl][i, h]
                                                      * np.exp(G[i] - G[j]))
            res = (np.eye(16) + R) @ im["Akk"][ch, h] - np.eye(16)
            assert np.abs(res).max() < 1e-12


# --------------------------------------------------------------------------
# Chunk quantities: product-of-decays form vs split-exponent form
# --------------------------------------------------------------------------

def test_chunk_quantities_split_exponent(oracle_mod):
    """The oracle forms D_{j+1:i} as products of per-token decays; the same
    quantities follow from the cumulative log-decay G by
    exp(G_i - G_j) = exp(G_i) exp(-G_j) ("K3's KDA precision problem", section
    on the per-channel decay in tiles).  Also checks the chunk numbering with
    a ragged last chunk."""
    T, H, d = 40, 2, 128
    inp = synthetic.make_inputs(1, T, H, 31)
    q, k, g, beta = (f64(inp[n])[0] for n in ("q", "k", "g", "beta"))
    im = oracle_mod.chunk_intermediates(inp["q"], inp["k"], inp["g"], inp["beta"], chunk=16)
    assert im["Akk"].shape[0] == 3
    s = 1 / math.sqrt(d)
    for ch in range(3):
        t0 = 16 * ch
        Cc = min(16, T - t0)
        for h in range(H):
            kh = _normalise(k[t0:t0 + Cc, h])
            qh = _normalise(q[t0:t0 + Cc, h])
            G = np.cumsum(g[t0:t0 + Cc, h], axis=0)
            E, Einv = np.exp(G), np.exp(-G)
            np.testing.assert_allclose(im["Kst"][ch, h, :Cc], E * kh, rtol=1e-13, atol=1e-300)
            np.testing.assert_allclose(im["Qst"][ch, h, :Cc], E * qh, rtol=1e-13, atol=1e-300)
            np.testing.assert_allclose(im["Kend"][ch, h, :Cc], kh * E[-1] * Einv,
                                       rtol=1e-12, atol=1e-300)
            np.testing.assert_allclose(im["D"][ch, h], E[-1], rtol=1e-13)
            Aqk = np.tril(s * (E * qh) @ (Einv * kh).T)
            R = np.tril(beta[t0:t0 + Cc, h][:, None] * ((E * kh) @ (Einv * kh).T), -1)
            np.testing.assert_allclose(im["Aqk"][ch, h, :Cc, :Cc], Aqk, rtol=1e-11, atol=1e-14)
            np.testing.assert_allclose(im["Akk"][ch, h, :Cc, :Cc],
                                       np.linalg.inv(np.eye(Cc) + R), rtol=1e-11, atol=1e-13)
            if Cc < 16:
                assert np.all(im["Kst"][ch, h, Cc:] == 0)
                np.testing.assert_array_equal(im["Akk"][ch, h, Cc:, Cc:], np.eye(16 - Cc))


def test_sigmoid_values(oracle_mod):
    """beta from a logit: the logistic function's fixed points and identities
    (sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, sigmoid(-x) = 1 - sigmoid(x),
    saturation without overflow) and scipy's expit on a spread of logits."""
    scipy_special = pytest.importorskip("scipy.special")
    y = oracle_mod.sigmoid(np.array([0.0, math.log(3.0), -math.log(3.0), -800.0, 800.0]))
    assert y[0] == 0.5
    assert abs(y[1] - 0.75) < 1e-15 and abs(y[2] - 0.25) < 1e-15
    assert y[3] == 0.0 and y[4] == 1.0
    x = np.random.default_rng(5).normal(0.0, 4.0, size=1000)
    y = oracle_mod.sigmoid(x)
    np.testing.assert_allclose(y, scipy_special.expit(x), rtol=1e-14, atol=0)
    np.testing.assert_allclose(oracle_mod.sigmoid(-x), 1.0 - y, rtol=0, atol=1e-15)


def test_beta_logit_path(oracle_mod):
    """beta_is_logit: the operation on logits equals the operation on
    sigmoid(logits) computed by scipy; logit 0 is beta = 1/2; a logit of -60
    (beta ~ 9e-27) is the beta = 0 closed form (pure decay) to rounding."""
    scipy_special = pytest.importorskip("scipy.special")
    inp = small_inputs(B=2, T=23, H=2, d=8, seed=11)
    q, k, v, g = map(f64, (inp["q"], inp["k"], inp["v"], inp["g"]))
    init = f64(inp["init_state"])
    logit = np.random.default_rng(2).normal(0.0, 2.0, size=(2, 23, 2))
    for form in ("kda_token", "kda_chunk"):
        fn = getattr(oracle_mod, form)
        o1, f1 = fn(q, k, v, g, logit, init, beta_is_logit=True)
        o2, f2 = fn(q, k, v, g, scipy_special.expit(logit), init)
        assert rel_fro(o1, o2) < 1e-13 and rel_fro(f1, f2) < 1e-13
    o1, f1 = oracle_mod.kda_token(q, k, v, g, np.zeros((2, 23, 2)), init, beta_is_logit=True)
    o2, f2 = oracle_mod.kda_token(q, k, v, g, np.full((2, 23, 2), 0.5), init)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(f1, f2)
    # -60: beta = 8.8e-27, so the state is S_0 Diag(exp(G_t)) to ~1e-25 of its
    # size (weak decay, so that the state stays of order one)
    g = 0.02 * g
    o1, f1 = oracle_mod.kda_token(q, k, v, g, np.full((2, 23, 2), -60.0), init,
                                  beta_is_logit=True)
    G = np.cumsum(g, axis=1)                                   # [B, T, H, dk]
    s = 1 / math.sqrt(8)
    qh = _normalise(q)
    for b in range(2):
        for h in range(2):
            S0 = init[b, h]
            expect = np.stack([s * (S0 * np.exp(G[b, t, h])[None, :]) @ qh[b, t, h]
                               for t in range(23)])
            assert rel_fro(o1[b, :, h], expect) < 1e-13
            assert rel_fro(f1[b, h], S0 * np.exp(G[b, -1, h])[None, :]) < 1e-13
