"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself -- a library routine it must reduce to, a closed form, an
invariant, or brute force on tiny inputs.  Source of the method: Osawa et al.,
"Large-Scale Distributed Second-Order Optimization Using Kronecker-Factored
Approximate Curvature for Deep Convolutional Neural Networks", section 3.2
(Eq. 3-7) and section 1 (diagonal BatchNorm Fisher)."""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def _spd(d, rng, scale=1.0):
    X = rng.standard_normal((d + 3, d))
    return scale * (X.T @ X) / (d + 3) + 0.1 * scale * np.eye(d)


# --------------------------------------------------------------- im2col / Eq.5

CONV_CASES = [
    # n, h, w, c, cout, k, stride, pad
    (2, 7, 6, 3, 4, 3, 1, 1),
    (1, 9, 9, 2, 3, 7, 2, 3),
    (2, 8, 8, 5, 2, 1, 2, 0),
    (3, 5, 5, 4, 3, 1, 1, 0),
    (1, 6, 7, 2, 2, 3, 2, 1),
]


def _flat_weight(W):
    # library weight [cout, c, kh, kw] -> patch-column order (r*kw + s)*c + ch
    cout, c, kh, kw = W.shape
    return W.transpose(0, 2, 3, 1).reshape(cout, kh * kw * c)


@pytest.mark.parametrize("case", CONV_CASES)
def test_im2col_is_the_library_convolution(case):
    """P W^T must equal a direct library convolution: pins the patch index,
    the padding value and the column order (Eq. 5's A is built on P)."""
    n, h, w, c, cout, k, s, p = case
    x = RNG.standard_normal((n, h, w, c))
    W = RNG.standard_normal((cout, c, k, k))
    P = oracle.im2col(x, k, k, (s, s), (p, p))
    y = P @ _flat_weight(W).T
    ref = torch.nn.functional.conv2d(torch.from_numpy(x).permute(0, 3, 1, 2),
                                     torch.from_numpy(W), stride=s, padding=p)
    ref = ref.permute(0, 2, 3, 1).reshape(-1, cout).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", CONV_CASES[:3])
def test_weight_grad_is_autograd(case):
    """grad = Gam^T P / n equals the autograd weight gradient of the mean
    over samples of <conv(x, W), g> (Eq. 1's E[.] is a mean over samples)."""
    n, h, w, c, cout, k, s, p = case
    x = RNG.standard_normal((n, h, w, c))
    W = torch.from_numpy(RNG.standard_normal((cout, c, k, k))).requires_grad_(True)
    y = torch.nn.functional.conv2d(torch.from_numpy(x).permute(0, 3, 1, 2), W, stride=s, padding=p)
    g = torch.from_numpy(RNG.standard_normal(tuple(y.shape)))
    ((y * g).sum() / n).backward()
    P = oracle.im2col(x, k, k, (s, s), (p, p))
    Gam = g.permute(0, 2, 3, 1).reshape(-1, cout).numpy()
    grad = oracle.weight_grad(P, Gam, n)
    np.testing.assert_allclose(grad, _flat_weight(W.grad.numpy()), rtol=1e-11, atol=1e-12)


def test_fc_bias_column_and_fc_as_conv():
    """FC with bias: P = [a, 1]; a 1x1 stride-1 conv equals FC on pixel rows;
    a k x k pad-0 conv on a k x k image equals FC on the flattened image."""
    a = RNG.standard_normal((6, 5))
    P = oracle.im2col(a, append_one=True)
    np.testing.assert_array_equal(P, np.concatenate([a, np.ones((6, 1))], axis=1))
    x = RNG.standard_normal((2, 3, 4, 5))
    np.testing.assert_array_equal(oracle.im2col(x), x.reshape(-1, 5))
    x = RNG.standard_normal((3, 3, 3, 2))
    np.testing.assert_array_equal(oracle.im2col(x, 3, 3), x.reshape(3, -1))


def test_gram_is_library_matmul_and_symmetric_psd():
    for M, d in [(1, 1), (7, 3), (50, 17), (5, 40)]:
        P = RNG.standard_normal((M, d))
        S = oracle.gram(P)
        np.testing.assert_allclose(S, P.T @ P, rtol=1e-12, atol=1e-12)
        assert np.array_equal(S, S.T)  # bitwise symmetric
        ev = np.linalg.eigvalsh(S)
        assert ev.min() >= -1e-12 * max(ev.max(), 1.0)


def test_gram_entries_match_full_statistic():
    x = RNG.standard_normal((2, 6, 5, 3))
    P = oracle.im2col(x, 3, 3, (1, 1), (1, 1), append_one=True)
    S = oracle.gram(P)
    d = P.shape[1]
    ii = RNG.integers(0, d, 40)
    jj = RNG.integers(0, d, 40)
    ii[:2] = d - 1
    e = oracle.gram_entries(x, ii, jj, 3, 3, (1, 1), (1, 1), append_one=True)
    np.testing.assert_allclose(e, S[ii, jj], rtol=1e-12, atol=1e-12)


def test_rank_one_factors_and_exact_fisher_at_batch_one():
    """FC at batch 1: A = a a^T, G = g g^T are rank one, and G (x) A equals the
    exact empirical Fisher vec(grad) vec(grad)^T of Eq. 3 with grad = g a^T."""
    a = RNG.standard_normal((1, 5))
    g = RNG.standard_normal((1, 4))
    P = oracle.im2col(a, append_one=True)
    A = oracle.factor_ema(np.zeros((6, 6)), P, 0.0)
    G = oracle.factor_ema(np.zeros((4, 4)), g, 0.0)
    evA = np.sort(np.linalg.eigvalsh(A))[::-1]
    evG = np.sort(np.linalg.eigvalsh(G))[::-1]
    np.testing.assert_allclose(evA[0], (P ** 2).sum(), rtol=1e-12)
    np.testing.assert_allclose(evG[0], (g ** 2).sum(), rtol=1e-12)
    assert np.abs(evA[1:]).max() < 1e-12 and np.abs(evG[1:]).max() < 1e-12
    grad = oracle.weight_grad(P, g, 1)          # = g^T [a, 1]
    v = grad.reshape(-1)
    np.testing.assert_allclose(np.kron(G, A), np.outer(v, v), rtol=1e-12, atol=1e-14)


def test_ema_closed_form_and_lower_bound():
    d, xi = 6, 0.95
    P = RNG.standard_normal((9, d))
    Fhat = (P.T @ P) / 9
    F = np.eye(d)
    for k in range(1, 6):
        F = oracle.factor_ema(F, P, xi)
        np.testing.assert_allclose(F, xi ** k * np.eye(d) + (1 - xi ** k) * Fhat,
                                   rtol=1e-12, atol=1e-13)
    F1 = oracle.factor_ema(np.eye(d), P, xi)
    assert np.linalg.eigvalsh(F1).min() >= xi - 1e-12


def test_chunked_accumulation_equals_one_statistic():
    """32 chunks of rows summed == the statistic of all rows (Osawa et al.
    section 2: gradient accumulation emulates a large mini-batch)."""
    P = RNG.standard_normal((32 * 5, 7))
    whole = oracle.gram(P)
    parts = sum(oracle.gram(P[i * 5:(i + 1) * 5]) for i in range(32))
    np.testing.assert_allclose(parts, whole, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ inversion / Eq.6

@pytest.mark.parametrize("d", [1, 2, 5, 33, 130])
def test_cholesky_trtri_lauum_match_library(d):
    A = _spd(d, RNG)
    U = oracle.cholesky_upper(A)
    np.testing.assert_allclose(U, np.linalg.cholesky(A).T, rtol=1e-10, atol=1e-12)
    assert np.all(np.tril(U, -1) == 0)
    V = oracle.trtri_upper(U)
    np.testing.assert_allclose(U @ V, np.eye(d), atol=1e-10)
    np.testing.assert_allclose(oracle.lauum_upper(V), V @ V.T, rtol=1e-12, atol=1e-13)
    for damp in (0.0, 1e-3, 0.5):
        Ai = oracle.damped_inverse(A, damp)
        R = (A + damp * np.eye(d)) @ Ai - np.eye(d)
        assert np.abs(R).max() < 1e-10
        np.testing.assert_allclose(Ai, np.linalg.inv(A + damp * np.eye(d)), rtol=1e-9, atol=1e-10)


def test_not_positive_definite_is_reported():
    with pytest.raises(np.linalg.LinAlgError):
        oracle.cholesky_upper(-np.eye(3))
    A = np.eye(4)
    A[2, 2] = 0.0
    with pytest.raises(np.linalg.LinAlgError, match="pivot 2"):
        oracle.damped_inverse(A, 0.0)


# ------------------------------------------------------- damping / Eq.6-7 pins

def test_pi_split_identity_closed_form():
    """A = I, G = I of different sizes: pi = 1, both damps are sqrt(gamma)."""
    da, dg = oracle.pi_damping(np.eye(7), np.eye(3), 1e-3)
    assert abs(da - np.sqrt(1e-3)) < 1e-15 and abs(dg - np.sqrt(1e-3)) < 1e-15
    da, dg = oracle.pi_damping(4.0 * np.eye(7), np.eye(3), 1e-3)   # pi = 2
    np.testing.assert_allclose([da, dg], [2 * np.sqrt(1e-3), np.sqrt(1e-3) / 2], rtol=1e-14)
    da, dg = oracle.pi_damping(4.0 * np.eye(7), np.eye(3), 1e-3, pi_split=False)
    assert da == dg == np.sqrt(1e-3)


@pytest.mark.parametrize("dA,dG", [(1, 1), (3, 2), (6, 5), (4, 4)])
def test_factored_preconditioner_is_explicit_kronecker_solve(dA, dG):
    """Eq. 6-7: G^-1 grad A^-1 == (G (x) A)^-1 vec(grad) (row-major vec),
    undamped (gamma = 0) and with the pi-split damping, where the damped
    product expands to A(x)G-form terms + gamma I."""
    rng = np.random.default_rng(dA * 10 + dG)
    A = _spd(dA, rng)
    G = _spd(dG, rng, scale=1e-3)
    grad = rng.standard_normal((dG, dA))
    # undamped
    out = oracle.precondition(oracle.damped_inverse(G, 0.0), grad, oracle.damped_inverse(A, 0.0))
    ref = np.linalg.solve(np.kron(G, A), grad.reshape(-1)).reshape(dG, dA)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())
    # pi-split damping
    gamma = 1e-3
    da, dg = oracle.pi_damping(A, G, gamma)
    assert abs(da * dg - gamma) < 1e-15
    K = (np.kron(G, A) + dg * np.kron(np.eye(dG), A) + da * np.kron(G, np.eye(dA))
         + gamma * np.eye(dA * dG))
    np.testing.assert_allclose(K, np.kron(G + dg * np.eye(dG), A + da * np.eye(dA)),
                               rtol=1e-12, atol=1e-15)
    out = oracle.precondition(oracle.damped_inverse(G, dg), grad, oracle.damped_inverse(A, da))
    ref = np.linalg.solve(K, grad.reshape(-1)).reshape(dG, dA)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())


def test_precondition_rows_are_rows_of_the_kronecker_solve():
    """Selected rows of Eq. 7 (the sampled check at sizes where the full
    product is too slow): equal to rows of the explicit Kronecker solve, in
    any order and with repeats."""
    rng = np.random.default_rng(11)
    dA, dG = 6, 5
    A, G = _spd(dA, rng), _spd(dG, rng, scale=1e-2)
    grad = rng.standard_normal((dG, dA))
    Ainv, Ginv = oracle.damped_inverse(A, 0.1), oracle.damped_inverse(G, 0.01)
    K = np.kron(G + 0.01 * np.eye(dG), A + 0.1 * np.eye(dA))
    ref = np.linalg.solve(K, grad.reshape(-1)).reshape(dG, dA)
    rows = [4, 0, 2, 2]
    got = oracle.precondition_rows(Ginv, grad, Ainv, rows)
    np.testing.assert_allclose(got, ref[rows], rtol=1e-9, atol=1e-12 * np.abs(ref).max())
    full = oracle.precondition(Ginv, grad, Ainv)
    np.testing.assert_allclose(got, full[rows], rtol=1e-12, atol=1e-15 * np.abs(full).max())


def test_pi_split_is_invariant_to_moving_scale_between_factors():
    """A -> cA, G -> G/c leaves the pi-damped preconditioned gradient
    unchanged (so the choice of which factor carries 1/M is immaterial)."""
    rng = np.random.default_rng(7)
    A, G = _spd(5, rng), _spd(3, rng, 1e-4)
    grad = rng.standard_normal((3, 5))
    outs = []
    for c in (1.0, 37.0, 1e-3):
        r = oracle.kfac_layer_step(c * A, G / c, np.zeros((1, 5)), np.zeros((1, 3)), grad,
                                   xi=1.0, gamma=1e-3)
        outs.append(r["precond"])
    np.testing.assert_allclose(outs[1], outs[0], rtol=1e-9)
    np.testing.assert_allclose(outs[2], outs[0], rtol=1e-9)


# ------------------------------------------------------------------- BN diag

def test_bn_diag_is_diagonal_of_explicit_fisher():
    x = RNG.standard_normal((11, 6))
    F, g, o = oracle.bn_diag_fisher(x, 1e-3)
    Ffull = sum(np.outer(r, r) for r in x) / 11
    np.testing.assert_allclose(F, np.diag(Ffull), rtol=1e-12)
    np.testing.assert_allclose(g, x.mean(axis=0), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(o, g / (F + 1e-3), rtol=1e-12)


def test_bn_constant_input_closed_form_and_ema():
    k = 0.25
    F, g, o = oracle.bn_diag_fisher(np.full((8, 3), k), 1e-3)
    np.testing.assert_allclose(F, k * k)
    np.testing.assert_allclose(g, k)
    np.testing.assert_allclose(o, k / (k * k + 1e-3))
    F, g, o = oracle.bn_diag_fisher(np.full((8, 3), k), 1e-3, xi=0.5, F=np.ones(3))
    np.testing.assert_allclose(F, 0.5 + 0.5 * k * k)
    np.testing.assert_allclose(o, k / (0.5 + 0.5 * k * k + 1e-3))


def test_fc_step_matches_stored_oracle_values():
    """Regression anchor: the single-FC-layer step as written by
    tests/golden/make_golden.py (oracle only)."""
    import json
    import os
    from tests.golden import make_golden
    ref = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fc64x32_step.json")))
    got = make_golden.summary(make_golden.compute())
    for k in ("damp_A", "damp_G"):
        assert abs(got[k] - ref[k]) <= 1e-13 * abs(ref[k])
    for k in ("A", "G", "Ainv", "Ginv", "precond", "grad"):
        assert abs(got[k]["fro"] - ref[k]["fro"]) <= 1e-12 * ref[k]["fro"]
        for (i, j, v), (_, _, w) in zip(got[k]["entries"], ref[k]["entries"]):
            assert abs(v - w) <= 1e-12 * max(abs(w), 1e-30) + 1e-300


# ------------------------------------------------------- Eq. 8 / stale schedule

def test_weight_update_closed_forms():
    rng = np.random.default_rng(21)
    w = rng.standard_normal((4, 6))
    P = rng.standard_normal((4, 6))
    np.testing.assert_array_equal(oracle.weight_update(w, P, 0.0), w)
    np.testing.assert_array_equal(oracle.weight_update(np.zeros_like(P), P, 1.0), -P)
    a = oracle.weight_update(w, P, 0.3)
    b = oracle.weight_update(w, P, 0.7)
    np.testing.assert_allclose(a + b - w, oracle.weight_update(w, P, 1.0), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("warmup,every,steps", [(0, 1, 7), (3, 4, 20), (10, 5, 8), (2, 10, 30)])
def test_refresh_schedule_closed_forms(warmup, every, steps):
    flags = [oracle.is_refresh_step(t, warmup, every) for t in range(steps)]
    assert all(flags[:warmup])
    if every == 1 or warmup >= steps:
        assert all(flags)
    after = max(0, steps - warmup)
    assert sum(flags) == min(warmup, steps) + (after + every - 1) // every


def test_stale_schedule_equals_stepwise_composition():
    """The schedule is the per-step composition of EMA, damping, inversion and
    preconditioning on refresh steps and preconditioning with the kept
    inverses otherwise."""
    rng = np.random.default_rng(22)
    steps = []
    for t in range(5):
        P = np.maximum(rng.standard_normal((12, 5)), 0)
        Gam = rng.standard_normal((12, 3)) * 1e-2
        steps.append((P, Gam, rng.standard_normal((3, 5)) * 1e-3))
    outs = oracle.kfac_schedule(np.eye(5), np.eye(3), steps, 0.95, 1e-3, warmup=1, every=3)
    A, G = np.eye(5), np.eye(3)
    for t, (P, Gam, grad) in enumerate(steps):
        if t in (0, 1, 4):   # warmup 1, every 3: steps 0, 1, 4 refresh
            A = oracle.factor_ema(A, P, 0.95)
            G = oracle.factor_ema(G, Gam, 0.95)
            da, dg = oracle.pi_damping(A, G, 1e-3)
            Ai, Gi = oracle.damped_inverse(A, da), oracle.damped_inverse(G, dg)
        np.testing.assert_allclose(outs[t], oracle.precondition(Gi, grad, Ai), rtol=1e-12)


# ------------------------------------------------------------- packed factor storage

def test_packed_upper_closed_form_and_round_trip():
    """Packed upper triangle (section 1: exploit the symmetry of the factors):
    for d = 3 the stored order is (0,0) (0,1) (0,2) (1,1) (1,2) (2,2); the
    position of (i, j) is i*d - i*(i+1)/2 + j, checked against an enumeration
    of the upper triangle; unpacking restores the symmetric matrix exactly."""
    F = np.array([[0.0, 1.0, 2.0], [1.0, 3.0, 4.0], [2.0, 4.0, 5.0]])
    np.testing.assert_array_equal(oracle.pack_upper(F), [0, 1, 2, 3, 4, 5])
    for d in (1, 2, 7, 64, 129):
        X = np.random.default_rng(d).standard_normal((d, d))
        S = X + X.T
        p = oracle.pack_upper(S)
        assert p.size == d * (d + 1) // 2
        pos = 0
        for i in range(d):
            for j in range(i, d):
                assert i * d - i * (i + 1) // 2 + j == pos
                assert p[pos] == S[i, j]
                pos += 1
        np.testing.assert_array_equal(oracle.unpack_upper(p, d), S)
        # only the upper triangle is read
        L = S.copy()
        L[np.tril_indices(d, -1)] = np.nan
        np.testing.assert_array_equal(oracle.pack_upper(L), p)
