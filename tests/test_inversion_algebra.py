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
  * the chain of one matrix: left-looking Cholesky block columns with
    lookahead (the diag kernel, the first panel block and the last term of
    the next diagonal update on the chain, the rest of each column and the
    earlier terms of the diagonal update after it as side work), the
    triangular inverse by recursive 2 x 2 blocking (T = L21 W11,
    W21 = -W22 T), bottom up by height, and the final product Wt Wt^T over
    upper tiles with K from each tile's first column (ktri), mirrored;
  * the same chain as launches on three streams (chain, side work, and the
    early triangular inverse whose nodes start once the Cholesky columns
    they read are done), executed in random and adversarial orders that
    keep only the dependencies the library declares.

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


def _dupd(c, j0, j1):
    """D_c -= L[c, j0:j1] L[c, j0:j1]^T (block columns j0 .. j1 - 1)."""
    return _job("L", c * NB, j0 * NB, "L", c * NB, j0 * NB, NB, NB, (j1 - j0) * NB, -1.0, 1.0, C=("D", c * NB, 0))


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
        if k + 2 < nb:   # X[k+2:, k+1] -= L[k+2:, :k+1] L[k+1, :k+1]^T, D_{k+2} -= L[k+2, :k+1] L[k+2, :k+1]^T
            side = [_job("L", kb + 2 * NB, 0, "L", kb + NB, 0, dp - kb - 2 * NB, NB, kb + NB, -1.0, 1.0,
                         C=("X", kb + 2 * NB, kb + NB)), _dupd(k + 2, 0, k + 1)]
        ops.append(("gemm", [_job("X", kb + NB, kb, "X", kb, kb, NB, NB, NB, 1.0, 0.0, C=("L", kb + NB, kb))],
                    side))
        # D_{k+1} -= L[k+1, k] L[k+1, k]^T (the earlier terms ran with the side work above)
        ops.append(("gemm", [_dupd(k + 1, k, k + 1)], []))
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


def _prep(buf, X0, dp):
    """The prep kernel: the blocks strictly below the diagonal 128-blocks into X
    (X's diagonal blocks and everything above them stay unwritten: NaN here),
    the diagonal blocks into D (lower part, zeros above)."""
    for bi in range(0, dp, NB):
        for bj in range(0, bi, NB):
            buf["X"][bi:bi + NB, bj:bj + NB] = X0[bi:bi + NB, bj:bj + NB]
        buf["D"][bi:bi + NB] = np.tril(X0[bi:bi + NB, bi:bi + NB])


def invert_like_the_library(F, damp, bn):
    d = F.shape[0]
    dp = -(-d // NB) * NB
    X0 = np.eye(dp)
    X0[:d, :d] = F + damp * np.eye(d)
    buf = {k: np.full((dp, dp), np.nan) for k in ("X", "W", "L")}
    buf["D"] = np.full((dp, NB), np.nan)
    _prep(buf, X0, dp)
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
    column, the first panel block and the last term of the next diagonal
    update between them, and 2 per level of the triangular inverse."""
    for dp, expect in ((128, 1), (256, 2 + 2 * 1 + 2), (1152, 9 + 2 * 8 + 2 * 4), (4608, 36 + 2 * 35 + 2 * 6)):
        assert len(chain(dp)) == expect, dp


# ---------------------------------------------------------------------------
# The same chain as launches on three streams, ordered only by what the
# library declares: each stream in order, a side launch after the op that
# enables it, an op after the side launch it names, every early-inverse step
# after the chain op it names, the final product after the last step.  Run in
# random and adversarial orders that respect exactly those edges, a missing
# edge shows up as a NaN read or a wrong inverse.

EARLY_TRI_MIN_NB = 8


def _t_job(o, n):
    h = NB * (n // NB // 2)
    return _job("L", o + h, o, "W", o, o, n - h, h, h, 1.0, 0.0, Ct=("L", o, o + h), ktri=True)


def _x_job(o, n):
    h = NB * (n // NB // 2)
    m = n - h
    return _job("X", o + h, o + h, "L", o, o + h, m, h, m, -1.0, 0.0, C=("X", o + h, o),
                Ct=("W", o, o + h), ktril=True)


def launch_graph(dp, early=True):
    """[(stream, kind, payload, deps)] in enqueue order; deps index earlier
    entries.  kind: "leaf" (payload: block offset) or "gemm" (payload: jobs)."""
    nb = dp // NB
    nodes, last = [], {}

    def add(stream, kind, payload, deps=()):
        d = set(deps)
        if stream in last:
            d.add(last[stream])
        nodes.append((stream, kind, payload, sorted(d)))
        last[stream] = len(nodes) - 1
        return len(nodes) - 1

    side_of, i_diag, i_first = {}, [None] * nb, [None] * nb

    def main(kind, payload, side=None, needs=None):
        i = add("main", kind, payload, [side_of[needs]] if needs is not None else [])
        if side:
            side_of[i] = add("side", "gemm", side, [i])
        return i

    last_side = None
    for k in range(nb):
        kb = k * NB
        side = None
        if k + 2 < nb:
            side = [_job("X", kb + 2 * NB, kb, "X", kb, kb, dp - kb - 2 * NB, NB, NB, 1.0, 0.0,
                         C=("L", kb + 2 * NB, kb))]
        i_diag[k] = main("leaf", kb, side)
        if side:
            last_side = i_diag[k]
        if k + 1 == nb:
            break
        side = None
        if k + 2 < nb:
            side = [_job("L", kb + 2 * NB, 0, "L", kb + NB, 0, dp - kb - 2 * NB, NB, kb + NB, -1.0, 1.0,
                         C=("X", kb + 2 * NB, kb + NB)), _dupd(k + 2, 0, k + 1)]
        i_first[k] = main("gemm", [_job("X", kb + NB, kb, "X", kb, kb, NB, NB, NB, 1.0, 0.0,
                                        C=("L", kb + NB, kb))], side, i_first[k - 1] if k >= 1 else None)
        if side:
            last_side = i_first[k]
        main("gemm", [_dupd(k + 1, k, k + 1)])
    fin_deps = []
    if early and nb >= EARLY_TRI_MIN_NB:
        def visit(o, n):
            if n == NB:
                return
            h = NB * (n // NB // 2)
            visit(o, h)
            add("tri", "gemm", [_t_job(o, n)], [i_first[min((o + h) // NB, nb - 2)]])
            visit(o + h, n - h)
            add("tri", "gemm", [_x_job(o, n)], [i_diag[(o + n) // NB - 1]])
        visit(0, dp)
        fin_deps = [last["tri"]]
    else:
        by_height = []
        _tri_nodes(0, dp, by_height)
        for ht in range(1, len(by_height)):
            main("gemm", [_t_job(o, n) for o, n in by_height[ht]], None, last_side if ht == 1 else None)
            main("gemm", [_x_job(o, n) for o, n in by_height[ht]])
        if len(by_height) <= 1 and last_side is not None:
            fin_deps = [side_of[last_side]]
    add("main", "fin", None, fin_deps)
    return nodes


def launch_graph_bulk(dp):
    """The chain with a third stream for the bulk of each column's update (the
    library's default): per block column k, after the diag launch, the side
    stream takes the panel L[k+2:, k] and the bulk stream, once that panel is
    done, the terms j <= k of column k + 2 (X[k+3:, k+2] and D_{k+2}); after
    the first panel block of k the side stream takes the last term of column
    k + 1 (K = 128) once column k + 1's bulk is done; the diagonal update on
    the chain waits for that bulk too.  Streams main / side / bulk."""
    nb = dp // NB
    nodes, last = [], {}

    def add(stream, kind, payload, deps=()):
        d = set(deps)
        if stream in last:
            d.add(last[stream])
        nodes.append((stream, kind, payload, sorted(d)))
        last[stream] = len(nodes) - 1
        return len(nodes) - 1

    side_of, bulk_of, i_diag, i_first = {}, {}, [None] * nb, [None] * nb

    def main(kind, payload, side=None, bulk=None, needs_side=None, needs_bulk=None, side_needs_bulk=None):
        deps = ([side_of[needs_side]] if needs_side is not None else []) + \
               ([bulk_of[needs_bulk]] if needs_bulk is not None else [])
        i = add("main", kind, payload, deps)
        if side:
            side_of[i] = add("side", "gemm", side, [i] + ([bulk_of[side_needs_bulk]]
                                                          if side_needs_bulk is not None else []))
        if bulk:
            bulk_of[i] = add("bulk", "gemm", bulk, [side_of[i]])
        return i

    last_side = last_bulk = None
    for k in range(nb):
        kb = k * NB
        side = bulk = None
        if k + 2 < nb:
            side = [_job("X", kb + 2 * NB, kb, "X", kb, kb, dp - kb - 2 * NB, NB, NB, 1.0, 0.0,
                         C=("L", kb + 2 * NB, kb))]
            bulk = [_dupd(k + 2, 0, k + 1)]
            if k + 3 < nb:   # X[k+3:, k+2] -= L[k+3:, :k+1] L[k+2, :k+1]^T
                bulk.insert(0, _job("L", kb + 3 * NB, 0, "L", kb + 2 * NB, 0, dp - kb - 3 * NB, NB, kb + NB,
                                    -1.0, 1.0, C=("X", kb + 3 * NB, kb + 2 * NB)))
        i_diag[k] = main("leaf", kb, side, bulk)
        if side:
            last_side = last_bulk = i_diag[k]
        if k + 1 == nb:
            break
        side = None
        bulk_k1 = i_diag[k - 1] if k >= 1 and k + 1 < nb else None   # column k + 1's bulk
        if k + 2 < nb:       # X[k+2:, k+1] -= L[k+2:, k] L[k+1, k]^T
            side = [_job("L", kb + 2 * NB, kb, "L", kb + NB, kb, dp - kb - 2 * NB, NB, NB, -1.0, 1.0,
                         C=("X", kb + 2 * NB, kb + NB))]
        i_first[k] = main("gemm", [_job("X", kb + NB, kb, "X", kb, kb, NB, NB, NB, 1.0, 0.0,
                                        C=("L", kb + NB, kb))], side,
                          needs_side=i_first[k - 1] if k >= 1 else None,
                          side_needs_bulk=bulk_k1 if side else None)
        if side:
            last_side = i_first[k]
        main("gemm", [_dupd(k + 1, k, k + 1)], needs_bulk=bulk_k1)
    by_height = []
    _tri_nodes(0, dp, by_height)
    for ht in range(1, len(by_height)):
        first = ht == 1
        main("gemm", [_t_job(o, n) for o, n in by_height[ht]], None, None,
             needs_side=last_side if first else None, needs_bulk=last_bulk if first else None)
        main("gemm", [_x_job(o, n) for o, n in by_height[ht]])
    fin_deps = []
    if len(by_height) <= 1 and last_side is not None:
        fin_deps = [side_of[last_side], bulk_of[last_bulk]]
    add("main", "fin", None, fin_deps)
    return nodes


def _emulated_inverse(F, damp, order):
    d = F.shape[0]
    dp = -(-d // NB) * NB
    X0 = np.eye(dp)
    X0[:d, :d] = F + damp * np.eye(d)
    buf = {k: np.full((dp, dp), np.nan) for k in ("X", "W", "L")}
    buf["D"] = np.full((dp, NB), np.nan)
    _prep(buf, X0, dp)
    out = None
    for kind, payload in order:
        if kind == "leaf":
            o = payload
            W = diag_block(buf["D"][o:o + NB])[1]
            buf["X"][o:o + NB, o:o + NB] = np.tril(W)
            buf["W"][o:o + NB, o:o + NB] = np.triu(W.T)
        elif kind == "gemm":
            results = []
            for j in payload:
                A = buf[j["A"]][j["ar"]:j["ar"] + j["M"], j["ac"]:j["ac"] + j["K"]]
                B = buf[j["B"]][j["br"]:j["br"] + j["N"], j["bc"]:j["bc"] + j["K"]]
                acc = np.full((j["M"], j["N"]), np.nan)
                for tm in range(0, j["M"], NB):
                    for tn in range(0, j["N"], NB):
                        k0 = tn if j["ktri"] else 0
                        k1 = min(j["K"], tm + NB) if j["ktril"] else j["K"]
                        acc[tm:tm + NB, tn:tn + NB] = A[tm:tm + NB, k0:k1] @ B[tn:tn + NB, k0:k1].T
                results.append((j, acc))
            for j, acc in results:
                if j["C"]:
                    b, r, c = j["C"]
                    old = buf[b][r:r + j["M"], c:c + j["N"]]
                    buf[b][r:r + j["M"], c:c + j["N"]] = j["alpha"] * acc + (j["beta"] * old if j["beta"] else 0.0)
                if j["Ct"]:
                    b, r, c = j["Ct"]
                    buf[b][r:r + j["N"], c:c + j["M"]] = (j["alpha"] * acc).T
        else:
            Wt = buf["W"]
            out = np.full((dp, dp), np.nan)
            for tm in range(0, dp, NB):
                for tn in range(tm, dp, NB):
                    tile = Wt[tm:tm + NB, tn:] @ Wt[tn:tn + NB, tn:].T
                    out[tm:tm + NB, tn:tn + NB] = tile
                    out[tn:tn + NB, tm:tm + NB] = tile.T
    return out[:d, :d]


def _orders(nodes, policy, seed):
    """A topological order of the launch graph: random, or the early-inverse
    and side streams as early (or the main stream as late) as the edges allow."""
    rng = np.random.default_rng(seed)
    done, order, left = set(), [], list(range(len(nodes)))
    rank = {"tri": 0, "bulk": 0, "side": 1, "main": 2}
    while left:
        ready = [i for i in left if all(d in done for d in nodes[i][3])]
        if policy == "random":
            i = ready[rng.integers(len(ready))]
        elif policy == "helpers_first":
            i = min(ready, key=lambda i: (rank[nodes[i][0]], i))
        else:  # main first
            i = min(ready, key=lambda i: (-rank[nodes[i][0]], i))
        left.remove(i)
        done.add(i)
        order.append((nodes[i][1], nodes[i][2]))
    return order


@pytest.mark.parametrize("early", [False, True])
@pytest.mark.parametrize("d", [1000, 1100, 1536])
@pytest.mark.parametrize("policy", ["random", "helpers_first", "main_first"])
def test_three_stream_schedule_respects_its_dependencies(d, policy, early):
    """The library's default keeps the triangular inverse on the chain
    (early=False: two streams); the early inverse is a build-time option."""
    rng = np.random.default_rng(d)
    Z = rng.standard_normal((d, d // 2))
    F = Z @ Z.T / (d // 2)
    damp = 0.05
    nodes = launch_graph(-(-d // NB) * NB, early=early)
    assert any(n[0] == "tri" for n in nodes) == early
    for seed in range(2 if policy == "random" else 1):
        inv = _emulated_inverse(F, damp, _orders(nodes, policy, seed))
        assert np.isfinite(inv).all()
        R = (F + damp * np.eye(d)) @ inv - np.eye(d)
        assert np.abs(R).max() < 1e-8


def test_early_inverse_graph_shape():
    """Main-stream launches of a 4608-wide matrix with the early inverse: 36
    diag launches, 35 first panel blocks, 35 last terms of the diagonal
    updates and the final product; the inverse's 35 nodes are 70 launches on
    the third stream."""
    nodes = launch_graph(4608, early=True)
    count = {}
    for n in nodes:
        count[n[0]] = count.get(n[0], 0) + 1
    assert count == {"main": 36 + 35 + 35 + 1, "side": 34 + 34, "tri": 70}
    # a matrix under the threshold keeps the inverse on its chain
    assert not any(n[0] == "tri" for n in launch_graph(896, early=True))


@pytest.mark.parametrize("d", [1, 200, 384, 1000, 1100, 1536])
@pytest.mark.parametrize("policy", ["random", "helpers_first", "main_first"])
def test_bulk_stream_schedule_respects_its_dependencies(d, policy):
    """The three-stream Cholesky (bulk of each column's update one column early
    on a stream of its own) in random and adversarial orders."""
    rng = np.random.default_rng(d + 7)
    Z = rng.standard_normal((d, max(d // 2, 1)))
    F = Z @ Z.T / max(d // 2, 1)
    damp = 0.05
    nodes = launch_graph_bulk(-(-d // NB) * NB)
    for seed in range(2 if policy == "random" else 1):
        inv = _emulated_inverse(F, damp, _orders(nodes, policy, seed))
        assert np.isfinite(inv).all()
        R = (F + damp * np.eye(d)) @ inv - np.eye(d)
        assert np.abs(R).max() < 1e-8


def _regions(kind, payload, dp):
    """(reads, writes) of one launch as (buffer, r0, r1, c0, c1) rectangles."""
    if kind == "leaf":
        o = payload
        return [("D", o, o + NB, 0, NB)], [("X", o, o + NB, o, o + NB), ("W", o, o + NB, o, o + NB)]
    if kind == "fin":
        return [("W", 0, dp, 0, dp)], []
    rd, wr = [], []
    for j in payload:
        rd.append((j["A"], j["ar"], j["ar"] + j["M"], j["ac"], j["ac"] + j["K"]))
        rd.append((j["B"], j["br"], j["br"] + j["N"], j["bc"], j["bc"] + j["K"]))
        if j["C"]:
            b, r, c = j["C"]
            wr.append((b, r, r + j["M"], c, c + j["N"]))
            if j["beta"]:
                rd.append((b, r, r + j["M"], c, c + j["N"]))
        if j["Ct"]:
            b, r, c = j["Ct"]
            wr.append((b, r, r + j["N"], c, c + j["M"]))
    return rd, wr


def _overlap(a, b):
    return a[0] == b[0] and a[1] < b[2] and b[1] < a[2] and a[3] < b[4] and b[3] < a[4]


def _races(nodes, dp):
    """Pairs of launches that touch a common region (one of them writing it)
    with no dependency path between them in either direction."""
    n = len(nodes)
    reach = [set() for _ in range(n)]      # reach[i]: nodes that must finish before i starts
    for i, nd in enumerate(nodes):
        for d in nd[3]:
            reach[i] |= reach[d] | {d}
    regs = [_regions(nd[1], nd[2], dp) for nd in nodes]
    out = []
    for i in range(n):
        for k in range(i):
            if k in reach[i] or i in reach[k]:
                continue
            ri, wi = regs[i]
            rk, wk = regs[k]
            if any(_overlap(a, b) for a in wi for b in rk + wk) or any(_overlap(a, b) for a in wk for b in ri):
                out.append((k, i))
    return out


@pytest.mark.parametrize("dp", [128, 384, 1024, 1536])
def test_launch_graphs_have_no_unordered_conflicting_launches(dp):
    """Every two launches that touch a common region, one writing it, are
    ordered by the declared dependencies (a check of the whole graph, which
    also covers the updates that commute and so pass any execution order)."""
    assert _races(launch_graph_bulk(dp), dp) == []
    assert _races(launch_graph(dp, early=False), dp) == []
