"""The damped inversion as the CUDA library schedules it, restated in float64
numpy and checked against numpy's inverse (no GPU).

Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
Kronecker-Factored Approximate Curvature ...", section 3.2, Eq. 6: each damped
factor X = F + damp I is inverted on its own.  The library inverts X through
its Cholesky factor X = L L^T: W = L^-1, then X^-1 = W^T W.  This file
restates, operation by operation and with the same buffer offsets:

  * the diag kernel, which turns the lower triangle of a 128 x 128 SPD
    block into L (blocked right-looking Cholesky by 16) and W = L^-1
    (blocked by rows of 16);
  * the chain of one matrix: left-looking Cholesky block columns (update,
    then the diag kernel, whose other CTAs form the panel below the block), the triangular inverse by recursive 2 x 2 blocking
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


DB = 16


def diag_block(S):
    """The diag kernel on the lower triangle of a 128 x 128 SPD block, blocked
    by 16: right-looking Cholesky (L_cc = chol(S_cc) column by column as the
    warp does it; L_ic = S_ic L_cc^-T; S_ij -= L_ic L_jc^T for i >= j past c,
    lower triangle only), then W = L^-1 by block rows (W_ii = L_ii^-1;
    W_ij = -W_ii sum_{t=j}^{i-1} L_it W_tj).  Returns (L, W)."""
    n = S.shape[0]
    M = np.tril(np.array(S, dtype=np.float64))
    for c in range(0, n, DB):
        e = c + DB
        B = M[c:e, c:e].copy()
        for q in range(DB):
            B[q, q] = np.sqrt(B[q, q])
            B[q + 1:, q] /= B[q, q]
            for j in range(q + 1, DB):
                B[j:, j] -= B[j:, q] * B[j, q]
        M[c:e, c:e] = np.tril(B)
        if e < n:
            Lcc = M[c:e, c:e]
            for q in range(DB):          # forward substitution, a row per thread
                M[e:, c + q] /= Lcc[q, q]
                M[e:, c + q + 1:e] -= np.outer(M[e:, c + q], Lcc[q + 1:, q])
            M[e:, e:] -= np.tril(M[e:, c:e] @ M[e:, c:e].T)
    L = np.tril(M)
    W = np.zeros_like(L)
    for b in range(0, n, DB):
        Lb = L[b:b + DB, b:b + DB]
        for q in range(DB):              # a thread per column of W_bb
            x = np.zeros(DB)
            for r in range(DB):
                x[r] = ((1.0 if r == q else 0.0) - Lb[r, :r] @ x[:r]) / Lb[r, r]
            W[b:b + DB, b + q] = x
    for i in range(DB, n, DB):
        for j in range(0, i, DB):
            T = L[i:i + DB, j:i] @ W[j:i, j:j + DB]
            W[i:i + DB, j:j + DB] = -W[i:i + DB, i:i + DB] @ T
    return L, W


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
    """Ops of one dp x dp matrix, in the library's order: ("leaf", k, side
    problems) for a diag kernel launch, ("gemm", problems, side problems) for
    an engine launch."""
    ops, nb = [], dp // NB
    # the lookahead form: the chain holds the diag launch of k, the first panel
    # block L[k+1, k] and the diagonal update of k + 1; the rest of each block
    # column is side work launched after them (the library runs it on a side
    # stream, ordered by events; here it runs right after its op)
    for k in range(nb):
        kb = k * NB
        side = []
        if k + 2 < nb:   # L[k+2:, k] = X[k+2:, k] W_kk^T
            side = [_job("X", kb + 2 * NB, kb, "X", kb, kb, dp - kb - 2 * NB, NB, NB, 1.0, 0.0,
                         C=("L", kb + 2 * NB, kb))]
        ops.append(("leaf", kb, side))
        if k + 1 == nb:
            break
        side = []
        if k + 2 < nb:   # X[k+2:, k+1] -= L[k+2:, :k+1] L[k+1, :k+1]^T
            side = [_job("L", kb + 2 * NB, 0, "L", kb + NB, 0, dp - kb - 2 * NB, NB, kb + NB, -1.0, 1.0,
                         C=("X", kb + 2 * NB, kb + NB))]
        ops.append(("gemm", [_job("X", kb + NB, kb, "X", kb, kb, NB, NB, NB, 1.0, 0.0, C=("L", kb + NB, kb))],
                    side))
        # D_{k+1} -= L[k+1, :k+1] L[k+1, :k+1]^T
        ops.append(("gemm", [_job("L", kb + NB, 0, "L", kb + NB, 0, NB, NB, kb + NB, -1.0, 1.0,
                                  C=("D", kb + NB, 0))], []))
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
    buf["D"] = np.full((dp, NB), np.nan)
    buf["X"][:] = np.tril(X0)                     # prep: lower part, zeros above
    for b in range(0, dp, NB):                     # ... and its diagonal blocks into D
        buf["D"][b:b + NB] = np.tril(X0)[b:b + NB, b:b + NB]
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
            W = diag_block(buf["D"][o:o + NB])[1]
            buf["X"][o:o + NB, o:o + NB] = np.tril(W)
            buf["W"][o:o + NB, o:o + NB] = np.triu(W.T)
            if op[2]:
                launch(op[2])
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


def test_diag_block_is_the_cholesky_factor_and_its_inverse():
    rng = np.random.default_rng(3)
    for scale in (0.01, 1e-4):
        Z = rng.standard_normal((NB, NB))
        S = Z @ Z.T / NB + scale * np.eye(NB)
        L, W = diag_block(S)
        Lr = np.linalg.cholesky(S)
        np.testing.assert_allclose(L, Lr, rtol=0, atol=1e-12)
        np.testing.assert_allclose(W, np.linalg.inv(Lr), rtol=1e-9, atol=1e-9)
        assert np.all(np.triu(W, 1) == 0.0) and np.all(np.triu(L, 1) == 0.0)
    # only the lower triangle is read
    Su = S.copy()
    Su[np.triu_indices(NB, 1)] = np.nan
    L2, W2 = diag_block(Su)
    assert np.array_equal(L2, L) and np.array_equal(W2, W)


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
    """Ops on the chain of one matrix: the diag launch of every 128-wide block
    column, the first panel block and the next diagonal update between them,
    and 2 per level of the triangular inverse."""
    for dp, expect in ((128, 1), (256, 2 + 2 * 1 + 2), (1152, 9 + 2 * 8 + 2 * 4), (4608, 36 + 2 * 35 + 2 * 6)):
        assert len(chain(dp)) == expect, dp
