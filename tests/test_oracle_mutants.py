"""The oracle pins must catch plausible mistakes.  Each case plants one
mistake (a wrong sign, a dropped term, a swapped or transposed index) in a
copy of the oracle's C source, builds it on the CPU, and checks that at least
one pin in test_oracle_pins fails against that build."""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kfac_oracle.c")

# (label, original text, planted mistake, pins expected to catch it)
MUTANTS = [
    ("im2col pad sign", "long hi = ho * sh - ph + r, wi = wo * sw - pw + s;",
     "long hi = ho * sh + ph + r, wi = wo * sw - pw + s;",
     [lambda: pins.test_im2col_is_the_library_convolution(pins.CONV_CASES[0])]),
    ("im2col kernel index transposed", "row[(r * kw + s) * c + ch]", "row[(s * kh + r) * c + ch]",
     [lambda: pins.test_im2col_is_the_library_convolution(pins.CONV_CASES[0])]),
    ("gram wrong operand", "acc += pi[m] * pj[m];", "acc += pi[m] * pi[m];",
     [pins.test_gram_is_library_matmul_and_symmetric_psd]),
    ("ema drops 1/M", "(1.0 - xi) * S[k] / (double)M", "(1.0 - xi) * S[k]",
     [pins.test_ema_closed_form_and_lower_bound]),
    ("weight grad divides by rows", "grad[o * dA + i] = acc / (double)nsamples;",
     "grad[o * dA + i] = acc / (double)M;",
     [lambda: pins.test_weight_grad_is_autograd(pins.CONV_CASES[0])]),
    ("pi drops the dimension normalisation", "sqrt((trA / (double)dA) / (trG / (double)dG))",
     "sqrt(trA / trG)", [pins.test_pi_split_identity_closed_form]),
    ("pi damping swapped", "*damp_A = pi * sg;", "*damp_A = sg / pi;",
     [pins.test_pi_split_is_invariant_to_moving_scale_between_factors]),
    ("cholesky update sign", "A[i * n + j] -= uki * A[k * n + j];",
     "A[i * n + j] += uki * A[k * n + j];",
     [lambda: pins.test_cholesky_trtri_lauum_match_library(5)]),
    ("trtri sign", "X[i * n + j] = -acc / U[i * n + i];", "X[i * n + j] = acc / U[i * n + i];",
     [lambda: pins.test_cholesky_trtri_lauum_match_library(5)]),
    ("lauum transposed operand", "acc += V[i * n + k] * V[j * n + k];",
     "acc += V[i * n + k] * V[k * n + j];",
     [lambda: pins.test_cholesky_trtri_lauum_match_library(5)]),
    ("precondition drops G^-1", "acc += Ginv[o * dG + k] * T[k * dA + j];",
     "acc += (k == o) * T[k * dA + j];",
     [lambda: pins.test_factored_preconditioner_is_explicit_kronecker_solve(3, 2)]),
    ("precondition rows transposed A^-1", "out[t * dA + j] += uk * Ainv[k * dA + j];",
     "out[t * dA + j] += uk * Ainv[j * dA + k] * (j == k ? 1.0 : 0.5);",
     [pins.test_precondition_rows_are_rows_of_the_kronecker_solve]),
    ("weight update sign", "w[o * dA + j] -= eta * P[o * dA + j];", "w[o * dA + j] += eta * P[o * dA + j];",
     [pins.test_weight_update_closed_forms]),
    ("refresh schedule off by one", "return (t - warmup) % every == 0;", "return (t - warmup + 1) % every == 0;",
     [lambda: pins.test_refresh_schedule_closed_forms(3, 4, 20),
      pins.test_stale_schedule_equals_stepwise_composition]),
    ("packed row skips the diagonal", "for (long j = i; j < d; ++j) out[t++] = F[i * d + j];",
     "for (long j = i; j < d; ++j) out[t++] = F[i * d + (j + 1) % d];",
     [pins.test_packed_upper_closed_form_and_round_trip]),
    ("bn unbiased variance", "double f = s2 / (double)ns;", "double f = s2 / (double)(ns - 1);",
     [pins.test_bn_diag_is_diagonal_of_explicit_fisher]),
    ("bn drops damping", "out[c] = gmean[c] / (F[c] + gamma);", "out[c] = gmean[c] / F[c];",
     [pins.test_bn_diag_is_diagonal_of_explicit_fisher]),
]


@pytest.mark.parametrize("label,orig,bad,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, label, orig, bad, checks):
    text = open(SRC).read()
    assert text.count(orig) == 1, f"mutation anchor not unique: {orig!r}"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(orig, bad))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", str(lib), str(src), "-lm"])
    caught = False
    with oracle.variant(str(lib)):
        for check in checks:
            try:
                check()
            except (AssertionError, Exception):
                caught = True
    assert caught, f"no pin caught the planted mistake: {label}"
