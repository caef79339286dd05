"""The block-step formulation of the TMEM-resident Gauss-Jordan leaf, restated
in float64 numpy and checked against numpy's inverse (no GPU).

Each 32-pivot block step K of the sweep is ONE rank-32 product
    A += (-C~) W~^T,   C~ = A[:, K] with rows K replaced by P - I,
                       W~ = P^-1 A[K, :] with columns K replaced by I + P^-1,
run in two parts, as the kernel does: first on the columns K (B rows
I + P^-1), which leaves -C P^-1 there; then on the other columns, with the
columns of W taken from that result through the sign-symmetric structure of
the sweep (a_ij = -a_ji exactly when one of i, j has been pivoted).  The 32 x 32
pivot block is inverted by the rotating single-pivot sweep of the kernel's
pivot warp.  This pins the algebra the kernel is built on (Osawa et al.,
"Large-Scale Distributed Second-Order Optimization Using Kronecker-Factored
Approximate Curvature ...", section 3.2, Eq. 6: the damped factors are
inverted exactly); the GPU parity tests pin the kernel itself.
"""
import numpy as np
import pytest


def pivot_block_inverse(P):
    """Gauss-Jordan inverse without pivoting, one pivot at a time, the row
    registers rotating by one column per pivot so that the pivot column is
    always position 0 (rows i != k: a_ij - f a_kj with f = a_i0 / a_kk; the
    pivot row takes f = 1 - 1 / a_kk)."""
    p = np.array(P, dtype=np.float64)
    n = p.shape[0]
    for k in range(n):
        pk = p[k].copy()
        inv = 1.0 / pk[0]
        f = p[:, 0] * inv
        f[k] = 1.0 - inv
        new = np.empty_like(p)
        new[:, :n - 1] = p[:, 1:] - f[:, None] * pk[None, 1:]
        new[:, n - 1] = -f
        new[k, n - 1] = inv
        p = new
    return p


def tmem_leaf(A, b=32):
    """The leaf's sweep on an SPD block (both triangles stored)."""
    A = np.array(A, dtype=np.float64)
    n = A.shape[0]
    eye = np.eye(b)
    for s in range(n // b):
        ks = s * b
        K = slice(ks, ks + b)
        C = A[:, K].copy()                        # pivot column panel
        Pinv = pivot_block_inverse(C[K, :])       # by the warp holding rows K
        Ct = C.copy()
        Ct[K, :] -= eye                           # C~ = C - E_K
        # part 1: the columns K, B rows = rows of I + P^-1
        A[:, K] += -Ct @ (eye + Pinv).T
        # rows outside K now hold -C P^-1; W[:, i] = +v (i pivoted) or -v (i after K)
        v = A[:, K]
        i = np.arange(n)
        Wt = np.where((i < ks)[:, None], v, -v)
        rest = np.ones(n, dtype=bool)
        rest[K] = False
        # part 2: every other column
        A[:, rest] += -Ct @ Wt[rest].T
    return A


def _spd(n, seed, ridge=1e-2):
    rng = np.random.default_rng(seed)
    X = np.maximum(rng.standard_normal((2 * n, n)), 0.0)
    return X.T @ X / (2 * n) + ridge * np.eye(n)


def test_pivot_block_inverse_is_the_inverse():
    P = _spd(32, 1)
    assert np.abs(pivot_block_inverse(P) @ P - np.eye(32)).max() < 1e-10


@pytest.mark.parametrize("n", [32, 64, 128, 256])
def test_block_steps_give_the_inverse(n):
    A = _spd(n, n)
    X = tmem_leaf(A)
    assert np.abs(A @ X - np.eye(n)).max() < 1e-8
    np.testing.assert_allclose(X, np.linalg.inv(A), rtol=1e-8, atol=1e-10)


def test_identity_padding_block():
    """diag(X, I): the padded identity rows come out as identity."""
    A = np.eye(128)
    A[:100, :100] = _spd(100, 7)
    X = tmem_leaf(A)
    np.testing.assert_allclose(X[100:, 100:], np.eye(28), atol=1e-12)
    np.testing.assert_allclose(X[:100, 100:], 0.0, atol=1e-12)
    np.testing.assert_allclose(X[:100, :100], np.linalg.inv(A[:100, :100]), rtol=1e-8, atol=1e-10)


def test_sign_symmetry_holds_between_steps():
    """The invariant the kernel relies on: after block step s, a_ij = -a_ji
    exactly when one of i, j is among the pivoted rows, a_ij = a_ji otherwise."""
    n, b = 128, 32
    A0 = _spd(n, 3)
    for steps in range(1, n // b):
        A = np.array(A0)
        eye = np.eye(b)
        for s in range(steps):
            ks = s * b
            K = slice(ks, ks + b)
            C = A[:, K].copy()
            Pinv = np.linalg.inv(C[K, :])
            Ct = C.copy()
            Ct[K, :] -= eye
            A[:, K] += -Ct @ (eye + Pinv).T
            v = A[:, K]
            i = np.arange(n)
            Wt = np.where((i < ks)[:, None], v, -v)
            rest = np.ones(n, dtype=bool)
            rest[K] = False
            A[:, rest] += -Ct @ Wt[rest].T
        piv = np.arange(n) < steps * b
        sign = np.where(piv[:, None] ^ piv[None, :], -1.0, 1.0)
        np.testing.assert_allclose(A, sign * A.T, rtol=1e-9, atol=1e-11)
