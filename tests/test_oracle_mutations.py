"""Plant plausible mistakes in a copy of the oracle and check the pins see them.

Each mutation edits one expression of ``oracle/kda_oracle.c`` in a temporary
copy, builds it, and runs the pins of ``test_oracle_pins`` against that build.
A mutation that no pin catches would mean the oracle is not pinned against
that kind of error.  Nothing here touches the real oracle build or a GPU.
"""

import os

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, exact text in kda_oracle.c, replacement)
MUTATIONS = [
    ("token_error_sign", "double u = b * (v[th * dv + r0 + r] - pred);",
     "double u = b * (v[th * dv + r0 + r] + pred);"),
    ("token_write_along_q", "for (int64_t c = 0; c < dk; ++c) s[c] += u * kh[c];",
     "for (int64_t c = 0; c < dk; ++c) s[c] += u * qh[c];"),
    ("token_read_with_k", "for (int64_t c = 0; c < dk; ++c) o += s[c] * qh[c];",
     "for (int64_t c = 0; c < dk; ++c) o += s[c] * kh[c];"),
    ("token_decay_value_rows", "for (int64_t c = 0; c < dk; ++c) s[c] *= alpha[c];",
     "for (int64_t c = 0; c < dk; ++c) s[c] *= alpha[r0 + r];"),
    ("token_decay_first_channel", "alpha[c] = exp(g[th * dk + c]);",
     "alpha[c] = exp(g[th * dk]);"),
    ("token_no_scale", "out[th * dv + r0 + r] = scale * o;", "out[th * dv + r0 + r] = o;"),
    ("token_norm_no_sqrt", "double inv = 1.0 / sqrt(ss + eps);", "double inv = 1.0 / (ss + eps);"),
    ("token_beta_of_previous_row", "const double b = beta[th];",
     "const double b = beta[th > 0 ? th - 1 : th];"),
    ("chunk_aqk_strict", "Aqk[i * Cc + j] = (j <= i) ? scale * rqk : 0.0;",
     "Aqk[i * Cc + j] = (j < i) ? scale * rqk : 0.0;"),
    ("chunk_r_beta_column", "R[i * Cc + j] = (j < i) ? betac[i] * rkk : 0.0;",
     "R[i * Cc + j] = (j < i) ? betac[j] * rkk : 0.0;"),
    ("chunk_kend_start_decay",
     "Kend[i * dk + c] = w->kh[i * dk + c] * w->Dpair[((Cc - 1) * C + i) * dk + c];",
     "Kend[i * dk + c] = w->kh[i * dk + c] * w->Dpre[i * dk + c];"),
    ("chunk_akk_transposed", "acc += E[r * C + j] * Akk[i * Cc + j];",
     "acc += E[r * C + j] * Akk[j * Cc + i];"),
    ("chunk_state_no_decay", "double acc = S[r * dk + c] * Dtot[c];",
     "double acc = S[r * dk + c];"),
    ("chunk_pair_decay_off_by_one",
     "p *= w->alpha[i * dk + c];\n                w->Dpair",
     "p *= w->alpha[(i - 1) * dk + c];\n                w->Dpair"),
    ("chunk_prefix_exclusive",
     "p *= w->alpha[i * dk + c];\n            w->Dpre[i * dk + c] = p;",
     "w->Dpre[i * dk + c] = p;\n            p *= w->alpha[i * dk + c];"),
    ("forward_subst_sign", "acc -= R[i * C + j] * X[j * C + m];",
     "acc += R[i * C + j] * X[j * C + m];"),
    ("neumann_first_factor_sign", "X[i * C + j] = ((i == j) ? 1.0 : 0.0) - L[i * C + j];",
     "X[i * C + j] = ((i == j) ? 1.0 : 0.0) + L[i * C + j];"),
    ("neumann_one_factor_short", "for (int64_t e = 2; e < C; e *= 2) {",
     "for (int64_t e = 2; e < C / 2; e *= 2) {"),
    ("sigmoid_sign", "y[i] = 1.0 / (1.0 + exp(-x[i]));", "y[i] = 1.0 / (1.0 + exp(x[i]));"),
    ("sigmoid_negative_branch", "y[i] = e / (1.0 + e);", "y[i] = 1.0 / (1.0 + e);"),
]


def _pin_suite(o):
    """Run the pins against oracle object ``o``; return the names that failed."""
    failed = []
    checks = [
        ("hand_token", lambda: [pins.test_hand_computed(o, c, "token")
                                for c in pins._hand_cases()]),
        ("hand_chunk3", lambda: [pins.test_hand_computed(o, c, "chunk3")
                                 for c in pins._hand_cases()]),
        ("beta0", lambda: pins.test_beta_zero_is_pure_decay(o)),
        ("readback", lambda: pins.test_exact_readback(o)),
        ("orthonormal", lambda: pins.test_orthonormal_keys_closed_form(o)),
        ("perm", lambda: pins.test_channel_permutations(o)),
        ("chunk_vs_token_16f", lambda: pins.test_chunkwise_matches_token(o, 16, "forward")),
        ("chunk_vs_token_32n", lambda: pins.test_chunkwise_matches_token(o, 32, "neumann")),
        ("inverse16", lambda: pins.test_unitri_inverse(o, 16)),
        ("inverse32", lambda: pins.test_unitri_inverse(o, 32)),
        ("split_exponent", lambda: pins.test_chunk_quantities_split_exponent(o)),
        ("sigmoid", lambda: pins.test_sigmoid_values(o)),
        ("beta_logit", lambda: pins.test_beta_logit_path(o)),
    ]
    for name, fn in checks:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_unmutated_copy_passes(tmp_path):
    src = tmp_path / "kda_oracle.c"
    src.write_text(open(SRC).read())
    lib = oracle.build(force=True, src=str(src), out=str(tmp_path / "lib.so"))
    assert _pin_suite(oracle.Variant(lib)) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation anchor for %s not unique in the oracle" % name
    src = tmp_path / "kda_oracle.c"
    src.write_text(text.replace(old, new))
    lib = oracle.build(force=True, src=str(src), out=str(tmp_path / "lib.so"))
    failed = _pin_suite(oracle.Variant(lib))
    assert failed, "no pin caught the planted mistake %s" % name
