"""The damped inversion as the CUDA library schedules it, restated in float64
numpy and checked against numpy's inverse (no GPU).

Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
Kronecker-Factored Approximate Curvature ...", section 3.2, Eq. 6: each damped
factor X = F + damp I is inverted on its own.  The library inverts X through
its Cholesky factor X = L L^T: W = L^-1, then X^-1 = W^T W.  This file
restates, operation by operation and with the same buffer offsets:

  * the diag kernel's sweep, which turns the lower triangle of a 128 x 128
    SPD block into W = L^-1 in place, 8 pivots per step (the single-pivot
    rules M_ij -= p_i y_j, M_ic = -p_i w, M_cj *= w, M_cc = w, with
    w = 1/sqrt(M_cc) and p_i = w M_ic, fused over the pivot block);
  * the chain of one matrix: left-looking Cholesky block columns (update,
    diag leaf, panel), the triangular inverse by recursive 2 x 2 blocking
    bottom up by height (T = L21 W11, W21 = -W22 T), and the final product
    Wt Wt^T over upper tiles with K from each tile's first column (ktri),
    mirrored.

Every buffer region the library never writes is NaN here, so a product that
reads one shows up as a NaN in the result; output tiles are 128 rows by 128,
64 or 32 columns as the engine may choose.  The GPU parity tests pin the
kernels themselves.
"""
import numpy as np
import pytest

NB = 128


def pivot_block(S):
    """The single-pivot rules applied to a square lower block alone (what each
    of the diag kernel's first 128 threads does with its 8 x 8 pivot block): W_K."""
    S = np.tril(np.array(S, dtype=np.float64))
    n = S.shape[0]
    for q in range(n):
        w = 1.0 / np.sqrt(S[q, q])
        p = np.where(np.arange(n) > q, S[:, q] * w, 0.0)
        for r in range(q + 1, n):
            S[r, :q] -= p[r] * w * S[q, :q]
            S[r, q] = -p[r] * w
            S[r, q + 1:r + 1] -= p[r] * p[q + 1:r + 1]
        S[q, :q] *= w
        S[q, q] = w
    return S


def diag_sweep(S, panel=8):
    """The diag kernel's sweep on the lower triangle of S, `panel` pivots
    K = {c .. c+panel-1} per step: W_K from the pivot block alone, then
    Z_j = W_K M[K][j] (j before K), W_K^T e_(j-c) (j in K), W_K M[j][K]
    (j past K); rows past K take M_ij = (j in K ? 0 : M_ij) - Z_i . Z_j
    (j <= i), rows K take Z_j (j before K) and W_K."""
    n = S.shape[0]
    M = np.tril(S).astype(np.float64)
    for c in range(0, n, panel):
        E = c + panel
        Wk = pivot_block(M[c:E, c:E])
        Zb = (Wk @ M[c:E, :c]).T          # j before K
        Zk = Wk.T                          # j in K: row j-c of W_K^T
        Zp = M[E:, c:E] @ Wk.T             # j past K
        Z = np.vstack([Zb, Zk, Zp])
        new = M.copy()
        low = np.tril(np.ones((n, n), dtype=bool))[E:]
        base = M[E:].copy()
        base[:, c:E] = 0.0
        new[E:] = np.where(low, base - Z[E:] @ Z.T, M[E:])
        new[c:E, :c] = Zb.T
        new[c:E, c:E] = Wk
        M = new
    return M


def _job(A, ar, ac, B, br, bc, M, N, K, alpha, beta, C=None, Ct=None, ktri=False, ktril=False):
    return dict(A=A, ar=ar, ac=ac, B=B, br=br, bc=bc, M=M, N=N, K=K, alpha=alpha, beta=beta, C=C, Ct=Ct,
                ktri=ktri, ktril=ktril)


def _tri_nodes(o, n, by_height):
    if n == NB:
        return 0
    h = NB * (n // NB // 2)
    ht = 1 + max(_tri_nodes(o, h, by_height), _tri_nodes(o + h, n - h, by_height))
    while len(by_height) <= ht:
        by_height.append([])
    by_height[ht].append((o, n))
    return ht


def chain(dp):
    """Ops of one dp x dp matrix, in the library's order (leaf or engine).
    An engine op may carry side problems (the lookahead update of column
    block k + 2 by panels 0 .. k), which the library launches on a second
    stream once the op is done and which finish before the chain's update of
    that column by its last panel."""
    ops, nb = [], dp // NB
    for k in range(nb):
        kb = k * NB
        if k > 0:   # X[k:, k] -= L[k:, k-1] L[k, k-1]^T   (the last panel's share)
            ops.append(("gemm", [_job("L", kb, kb - NB, "L", kb, kb - NB, dp - kb, NB, NB, -1.0, 1.0,
                                      C=("X", kb, kb))], []))
        ops.append(("leaf", kb))
        if k + 1 < nb:   # L[k+1:, k] = X[k+1:, k] W_kk^T
            side = []
            if k + 2 < nb:   # X[k2:, k2] -= L[k2:, :k+1] L[k2, :k+1]^T
                k2b = (k + 2) * NB
                side = [_job("L", k2b, 0, "L", k2b, 0, dp - k2b, NB, kb + NB, -1.0, 1.0, C=("X", k2b, k2b))]
            ops.append(("gemm", [_job("X", kb + NB, kb, "X", kb, kb, dp - kb - NB, NB, NB, 1.0, 0.0,
                                      C=("L", kb + NB, kb))], side))
    by_height = []
    _tri_nodes(0, dp, by_height)
    for ht in range(1, len(by_height)):
        t, x = [], []
        for o, n in by_height[ht]:
            h = NB * (n // NB // 2)
            m = n - h
            t.append(_job("L", o + h, o, "W", o, o, m, h, h, 1.0, 0.0, Ct=("L", o, o + h), ktri=True))
            x.append(_job("X", o + h, o + h, "L", o, o + h, m, h, m, -1.0, 0.0, C=("X", o + h, o),
                          Ct=("W", o, o + h), ktril=True))
        ops.append(("gemm", t, []))
        ops.append(("gemm", x, []))
    return ops


def invert_like_the_library(F, damp, bn):
    d = F.shape[0]
    dp = -(-d // NB) * NB
    X0 = np.eye(dp)
    X0[:d, :d] = F + damp * np.eye(d)
    buf = {k: np.full((dp, dp), np.nan) for k in ("X", "W", "L")}
    buf["X"][:] = np.tril(X0)                     # prep: lower part, zeros above
    def launch(jobs):
        results = []
        for j in jobs:   # every problem of one launch reads before any writes
            A = buf[j["A"]][j["ar"]:j["ar"] + j["M"], j["ac"]:j["ac"] + j["K"]]
            B = buf[j["B"]][j["br"]:j["br"] + j["N"], j["bc"]:j["bc"] + j["K"]]
            acc = np.full((j["M"], j["N"]), np.nan)
            for tm in range(0, j["M"], NB):
                for tn in range(0, j["N"], bn):
                    k0 = tn if j["ktri"] else 0                       # B[j][t] = 0 for t < j
                    k1 = min(j["K"], tm + NB) if j["ktril"] else j["K"]  # A[i][t] = 0 for t > i
                    acc[tm:tm + NB, tn:tn + bn] = A[tm:tm + NB, k0:k1] @ B[tn:tn + bn, k0:k1].T
            results.append((j, acc))
        for j, acc in results:
            if j["C"]:
                b, r, c = j["C"]
                old = buf[b][r:r + j["M"], c:c + j["N"]]
                buf[b][r:r + j["M"], c:c + j["N"]] = j["alpha"] * acc + (j["beta"] * old if j["beta"] else 0.0)
            if j["Ct"]:
                b, r, c = j["Ct"]
                buf[b][r:r + j["N"], c:c + j["M"]] = (j["alpha"] * acc).T

    for op in chain(dp):
        if op[0] == "leaf":
            o = op[1]
            W = diag_sweep(buf["X"][o:o + NB, o:o + NB])
            buf["X"][o:o + NB, o:o + NB] = np.tril(W)
            buf["W"][o:o + NB, o:o + NB] = np.triu(W.T)
            continue
        launch(op[1])
        if op[2]:
            launch(op[2])
    Wt = buf["W"]
    out = np.full((dp, dp), np.nan)
    for tm in range(0, dp, NB):
        for tn in range(tm, dp, bn):   # upper tiles, K from the tile's first column, mirrored
            tile = Wt[tm:tm + NB, tn:] @ Wt[tn:tn + bn, tn:].T
            out[tm:tm + NB, tn:tn + bn] = tile
            out[tn:tn + bn, tm:tm + NB] = tile.T
    return out[:d, :d]


@pytest.mark.parametrize("n", [4, 8, 32])
def test_pivot_block_rules_are_the_inverse_cholesky_factor(n):
    rng = np.random.default_rng(4)
    Z = rng.standard_normal((n, n))
    S = Z @ Z.T / n + 0.1 * np.eye(n)
    np.testing.assert_allclose(pivot_block(S), np.linalg.inv(np.linalg.cholesky(S)), rtol=0, atol=1e-10)


def test_diag_sweep_is_the_inverse_cholesky_factor():
    rng = np.random.default_rng(3)
    Z = rng.standard_normal((NB, NB))
    S = Z @ Z.T / NB + 0.01 * np.eye(NB)
    for panel in (4, 8, 32):
        W = diag_sweep(S, panel)
        np.testing.assert_allclose(np.tril(W), np.linalg.inv(np.linalg.cholesky(S)), rtol=0, atol=1e-11)
    assert np.all(np.triu(W, 1) == 0.0)


@pytest.mark.parametrize("bn", [128, 64, 32])
@pytest.mark.parametrize("d", [1, 5, 128, 129, 300, 640])
def test_chain_inverts_and_reads_only_written_regions(d, bn):
    rng = np.random.default_rng(d)
    Z = rng.standard_normal((d, max(d // 3, 1)))
    F = Z @ Z.T / max(d // 3, 1)                   # rank-deficient PSD, like a raw factor statistic
    damp = 0.03
    inv = invert_like_the_library(F, damp, bn)
    assert np.isfinite(inv).all()
    R = (F + damp * np.eye(d)) @ inv - np.eye(d)
    assert np.abs(R).max() < 1e-8
    assert np.array_equal(inv, inv.T)


def test_chain_launch_counts():
    """Ops per matrix: 3 per 128-wide block column (minus the first update and
    the last panel) and 2 per level of the triangular inverse."""
    for dp, expect in ((128, 1), (256, 4 + 2), (1152, 9 * 3 - 2 + 2 * 4), (4608, 36 * 3 - 2 + 2 * 6)):
        assert len(chain(dp)) == expect, dp
