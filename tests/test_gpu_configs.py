"""GPU parity at the full sizes of the five workload configurations.

The single FC layer in fp32 is `test_gpu_parity.test_fc64x32_fp32_step`.  The
others run here on the same seeded inputs as the benchmark, in the launch
configuration it times (one batched call per phase):

  3x3 conv, 256 channels   the whole layer step against the oracle's whole
                           layer step (factors, inverses, preconditioned
                           gradient compared in full);
  ResNet-50 layer set      factor entries recomputed by the oracle straight
  FC 4096 -> 4096 + bias   from the inputs (sampled); on layers of every
                           kind, the damping, the FULL inverses and the
                           preconditioned gradient (full, or sampled rows at
                           FC 4096) against the oracle run on the factors the
                           kernels produced (so the bf16 error of the factor
                           statistic is not counted twice);
  1024-sample accumulation 32 chunks of 32 on representative layers (checked
                           as above), and the BN diagonal Fisher of all 53
                           BN layers in full;
  hard-conditioned         raw statistics (xi = 0) of the 2049-, 4097- and
  inversions               4608-wide factors damped by sqrt(gamma) alone
                           (condition numbers ~1e4) and by the pi split.

Tolerances (relative Frobenius error of the compared set unless stated):
factors and preconditioned gradients from bf16 inputs <= 2e-2; damped
inverses max |(F + damp I) inv - I| <= 1e-3, and <= 1e-3 relative to the
oracle's inverse of the same factor where the factor is well conditioned.
"""
import numpy as np
import pytest
import torch

import oracle
from second_order_optimisation_gb300 import kfac, workloads
from second_order_optimisation_gb300.step import KfacStep

pytestmark = pytest.mark.gpu
DEV = "cuda"
XI, GAMMA = 0.95, 1e-3


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def grad_dev(w):
    """grad[dG, dA] on the device with a leading dimension rounded up to 8
    (the bf16 preconditioner reads rows in 16-byte pieces), as a view."""
    dG, dA = w.shape
    buf = torch.zeros(dG, (dA + 7) // 8 * 8, dtype=w.dtype, device=DEV)
    buf[:, :dA] = w.to(DEV)
    return buf[:, :dA]


def sym_from_upper(U):
    U = np.triu(U)
    return U + np.triu(U, 1).T


def upper_samples(d, n, tag):
    """n seeded index pairs i <= j of a d x d matrix, corners included."""
    rng = np.random.default_rng(workloads.seed_of("samples", tag, d))
    i = rng.integers(0, d, n)
    j = rng.integers(0, d, n)
    ii = np.minimum(i, j).tolist() + [0, d - 1, 0]
    jj = np.maximum(i, j).tolist() + [0, d - 1, d - 1]
    return np.asarray(ii, dtype=np.int64), np.asarray(jj, dtype=np.int64)


def check_factor_samples(F, x, M, k=1, stride=1, pad=0, append_one=False, tag="", n=96):
    """Sampled entries of F = xi I + (1 - xi)/M P^T P (the EMA from I) against
    the oracle's entries of P^T P computed from the input itself; the factor,
    and the statistic alone on the off-diagonal samples, must be within 2e-2."""
    d = F.shape[0]
    ii, jj = upper_samples(d, n, tag)
    S = oracle.gram_entries(x, ii, jj, k, k, (stride, stride), (pad, pad), append_one)
    got = f64(F)[ii, jj]
    ref = XI * (ii == jj) + (1.0 - XI) / M * S
    assert rel(got, ref) <= 2e-2, (tag, rel(got, ref))
    off = ii != jj  # on the diagonal the statistic can sit below fp32 resolution of xi
    stat = got[off] * M / (1.0 - XI)
    assert rel(stat, S[off]) <= 2e-2, (tag, "statistic", rel(stat, S[off]))


def check_inverse_columns(F, Finv, damp, tag="", n=6):
    """max |(F + damp I) inv - I| over sampled columns (F read from its upper triangle)."""
    Fs = sym_from_upper(f64(F))
    d = Fs.shape[0]
    cols = np.unique(np.r_[0, d - 1, np.random.default_rng(workloads.seed_of("cols", tag, d)).integers(0, d, n)])
    inv = f64(Finv)[:, cols]
    R = Fs @ inv + damp * inv
    R[cols, np.arange(len(cols))] -= 1.0
    assert np.abs(R).max() <= 1e-3, (tag, np.abs(R).max())


def check_against_oracle(step, i, w, tag="", rows=None):
    """Damping, full inverses and the preconditioned gradient of layer i
    against the oracle run on the factors the kernels produced (upper
    triangles as stored, widened exactly): pi-split damping (rtol 1e-3),
    inverses relative to the oracle's Cholesky-based inverse (<= 1e-3), and
    G^-1 grad A^-1 with the oracle's inverses and the stored bf16 gradient
    (<= 2e-2; all rows, or the sampled `rows`)."""
    s = step.state[i]
    A = sym_from_upper(f64(s.A))
    G = sym_from_upper(f64(s.G))
    da, dg = oracle.pi_damping(A, G, GAMMA)
    dm = f64(step.damp)
    np.testing.assert_allclose(dm[2 * i:2 * i + 2], [da, dg], rtol=1e-3, err_msg=tag)
    Ainv = oracle.damped_inverse(A, da)
    Ginv = oracle.damped_inverse(G, dg)
    assert rel(f64(s.A_inv), Ainv) <= 1e-3, (tag, "A_inv", rel(f64(s.A_inv), Ainv))
    assert rel(f64(s.G_inv), Ginv) <= 1e-3, (tag, "G_inv", rel(f64(s.G_inv), Ginv))
    gr = f64(w)
    if rows is None:
        ref, got = oracle.precondition(Ginv, gr, Ainv), f64(s.out)
    else:
        ref, got = oracle.precondition_rows(Ginv, gr, Ainv, rows), f64(s.out)[rows]
    assert rel(got, ref) <= 2e-2, (tag, "precond", rel(got, ref))


# ------------------------------------------------- one 3x3 conv layer, full

def test_config_conv3x3_256_layer_step():
    """3x3 conv, 256 -> 256 channels, 14x14, batch 32 (6272 patch rows): the
    whole layer step (factors from I with xi = 0.95, pi-split damping with
    gamma = 1e-3, inversion, preconditioning) against the oracle's."""
    L = workloads.conv_3x3_256()
    x, g, w = workloads.layer_inputs(L, 32, "cfg-conv3x3")
    step = KfacStep([L], 32, xi=XI, gamma=GAMMA)
    step.run([x.to(DEV)], [g.to(DEV)], [grad_dev(w)])
    torch.cuda.synchronize()
    assert step.info.cpu().tolist() == [0, 0]
    s = step.state[0]
    P = oracle.im2col(x.float().numpy(), 3, 3, (1, 1), (1, 1))
    ref = oracle.kfac_layer_step(np.eye(L.d_a), np.eye(L.d_g), P, g.float().numpy(), w.float().numpy(),
                                 xi=XI, gamma=GAMMA)
    assert rel(np.triu(f64(s.A)), np.triu(ref["A"])) <= 2e-2
    assert rel(np.triu(f64(s.G)), np.triu(ref["G"])) <= 2e-2
    dm = f64(step.damp)
    np.testing.assert_allclose(dm, [ref["damp_A"], ref["damp_G"]], rtol=1e-3)
    for F, inv, dmp in ((s.A, s.A_inv, dm[0]), (s.G, s.G_inv, dm[1])):
        Fs = sym_from_upper(f64(F))
        R = (Fs + dmp * np.eye(Fs.shape[0])) @ f64(inv) - np.eye(Fs.shape[0])
        assert np.abs(R).max() <= 1e-3, np.abs(R).max()
    assert rel(f64(s.out), ref["precond"]) <= 2e-2, rel(f64(s.out), ref["precond"])


# ------------------------------------------------- ResNet-50 layer set, sampled

SAMPLED_LAYERS = ("conv1", "s1b1_3x3", "s2b1_3x3", "s2b1_proj", "s3b1_1x1a", "s4b3_3x3", "fc")


def _check_layer(step, i, x, g, w, M, tag):
    s = step.state[i]
    L = s.layer
    xa = x.float().numpy()
    if L.hin == 1 and L.k == 1:
        xa = xa.reshape(xa.shape[0], -1)
    check_factor_samples(s.A, xa, M, L.k, L.stride, L.pad, L.bias, tag=f"{tag}{L.name}A")
    check_factor_samples(s.G, g.float().numpy(), M, tag=f"{tag}{L.name}G")
    dm = f64(step.damp)
    check_inverse_columns(s.A, s.A_inv, dm[2 * i], tag=f"{tag}{L.name}A")
    check_inverse_columns(s.G, s.G_inv, dm[2 * i + 1], tag=f"{tag}{L.name}G")
    rows = None
    if L.d_g * L.d_a > 4_000_000:   # FC 4096: sampled rows of Eq. 7
        rows = np.unique(np.r_[0, L.d_g - 1, np.random.default_rng(
            workloads.seed_of("pcrows", tag, L.name)).integers(0, L.d_g, 30)])
    check_against_oracle(step, i, w, tag=f"{tag}{L.name}", rows=rows)


def test_config_resnet50_step_sampled():
    """All 54 layers at batch 32 in one call per phase, as the benchmark runs
    them; sampled checks on layers covering every kind of source (7x7 stride-2
    patches, 3x3 taps through the im2col map, stride-2 3x3 and 1x1, direct
    1x1, the 4608-wide factor, FC with bias)."""
    layers = workloads.resnet50_layers()
    step = KfacStep(layers, 32, xi=XI, gamma=GAMMA)
    xs, gs, ws, keep = [], [], [], {}
    for L in layers:
        x, g, w = workloads.layer_inputs(L, 32, "cfg-resnet50")
        xs.append(x.to(DEV))
        gs.append(g.to(DEV))
        ws.append(grad_dev(w))
        if L.name in SAMPLED_LAYERS:
            keep[L.name] = (x, g, w)
    step.run(xs, gs, ws)
    torch.cuda.synchronize()
    assert int(step.info.abs().sum().item()) == 0
    for i, L in enumerate(layers):
        if L.name in keep:
            x, g, w = keep[L.name]
            _check_layer(step, i, x, g, w, L.rows(32), "r50")


def test_config_fc4096_sampled():
    """FC 4096 -> 4096 with bias over 8192 rows: A is 4097 x 4097, G 4096 x 4096."""
    L = workloads.fc_4096()
    x, g, w = workloads.layer_inputs(L, 8192, "cfg-fc4096")
    step = KfacStep([L], 8192, xi=XI, gamma=GAMMA)
    step.run([x.to(DEV)], [g.to(DEV)], [grad_dev(w)])
    torch.cuda.synchronize()
    assert step.info.cpu().tolist() == [0, 0]
    _check_layer(step, 0, x, g, w, 8192, "fc4096")


# ------------------------------------- 1024-sample accumulation, BN Fisher

ACCUM_LAYERS = ("conv1", "s1b1_3x3", "s3b2_3x3", "s4b1_proj", "fc")


def test_config_accumulation_1024_in_32_chunks():
    """Factors accumulated over a 1024-sample mini-batch in 32 chunks of 32
    (beta = xi on the first chunk, 1 after; alpha = (1 - xi) / rows of all
    chunks), then damped, inverted and applied."""
    layers = [L for L in workloads.resnet50_layers() if L.name in ACCUM_LAYERS]
    step = KfacStep(layers, 32, xi=XI, gamma=GAMMA)
    chunks = 32
    rows_total = [L.rows(32) * chunks for L in layers]
    samples = {}
    for c in range(chunks):
        xs, gs = [], []
        for L in layers:
            x, g, _ = workloads.layer_inputs(L, 32, "cfg-accum", c, grad_w=False)
            xs.append(x.to(DEV))
            gs.append(g.to(DEV))
            xa = x.float().numpy()
            if L.hin == 1 and L.k == 1:
                xa = xa.reshape(xa.shape[0], -1)
            for fac, src, geo in (("A", xa, (L.k, L.stride, L.pad, L.bias)), ("G", g.float().numpy(), (1, 1, 0, False))):
                d = L.d_a if fac == "A" else L.d_g
                ii, jj = upper_samples(d, 96, f"acc{L.name}{fac}")
                k, st, p, b = geo
                S = oracle.gram_entries(src, ii, jj, k, k, (st, st), (p, p), b)
                key = (L.name, fac)
                samples[key] = samples.get(key, 0.0) + S
        step.factor_update(xs, gs, rows_total=rows_total, first=(c == 0))
    ws = [workloads.layer_inputs(L, 32, "cfg-accum", "w")[2] for L in layers]
    step.damp_invert()
    step.precondition([grad_dev(w) for w in ws])
    torch.cuda.synchronize()
    assert int(step.info.abs().sum().item()) == 0
    dm = f64(step.damp)
    for i, (L, M) in enumerate(zip(layers, rows_total)):
        s = step.state[i]
        for fac, F in (("A", s.A), ("G", s.G)):
            d = F.shape[0]
            ii, jj = upper_samples(d, 96, f"acc{L.name}{fac}")
            S = samples[(L.name, fac)]
            got = f64(F)[ii, jj]
            ref = XI * (ii == jj) + (1.0 - XI) / M * S
            assert rel(got, ref) <= 2e-2, (L.name, fac, rel(got, ref))
            off = ii != jj
            stat = got[off] * M / (1.0 - XI)
            assert rel(stat, S[off]) <= 2e-2, (L.name, fac, "statistic", rel(stat, S[off]))
        check_inverse_columns(s.A, s.A_inv, dm[2 * i], tag=f"acc{L.name}A")
        check_inverse_columns(s.G, s.G_inv, dm[2 * i + 1], tag=f"acc{L.name}G")
        check_against_oracle(step, i, ws[i], tag=f"acc{L.name}")


def test_config_bn_diag_fisher_all_53_layers():
    """Diagonal Fisher of the scale and shift of all 53 BN layers from
    per-sample gradients [1024, C] ~ N(0, 0.01^2), damped with gamma = 1e-3."""
    chans = workloads.resnet50_bn_channels()
    assert len(chans) == 53
    grads = workloads.bn_grads(chans, 1024, "cfg-bn")
    items, refs = [], []
    for xg, xb in grads:
        for x in (xg, xb):
            C = x.shape[1]
            items.append(kfac.BnItem(torch.from_numpy(x).to(DEV), torch.zeros(C, device=DEV),
                                     torch.empty(C, device=DEV), torch.empty(C, device=DEV)))
            refs.append(oracle.bn_diag_fisher(x, GAMMA))
    kfac.kfac_bn_diag_fisher(items, GAMMA, xi=0.0)
    torch.cuda.synchronize()
    for it, (Fo, go, po) in zip(items, refs):
        assert rel(f64(it.F), Fo) <= 1e-4
        assert rel(f64(it.precond), po) <= 1e-4


# ------------------------------------------------- hard-conditioned inversions

HARD_CASES = {
    # d = 2049: ResNet-50's FC layer (2048 -> 1000 + bias) at batch 32: the
    #           raw statistic has rank <= 32
    "fc2049": (lambda: [L for L in workloads.resnet50_layers() if L.name == "fc"][0], 32),
    # d = 4097: FC 4096 -> 4096 + bias over 8192 rows
    "fc4097": (workloads.fc_4096, 8192),
    # d = 4608: the last 3x3 conv (512 channels, 7x7) at batch 32: rank <= 1568
    "conv4608": (lambda: [L for L in workloads.resnet50_layers() if L.name == "s4b3_3x3"][0], 32),
}


@pytest.mark.parametrize("case", sorted(HARD_CASES))
def test_hard_conditioned_inversion(case):
    """Raw statistics (xi = 0: beta = 0, alpha = 1/M) of the widest factors,
    damped by sqrt(gamma) on each factor (pi_split = 0; lambda_max / damp of
    A ~ 1e4) and by the pi split: max |(F + damp I) inv - I| <= 1e-3 in both,
    the inverse of the well-conditioned pi-split A within 1e-3 of the
    oracle's, and the damping values equal to the oracle's."""
    make, batch = HARD_CASES[case]
    L = make()
    x, g, _ = workloads.layer_inputs(L, batch, "hard", case, grad_w=False)
    step = KfacStep([L], batch, xi=0.0, gamma=GAMMA)
    step.factor_update([x.to(DEV)], [g.to(DEV)])
    s = step.state[0]
    A = sym_from_upper(f64(s.A))
    G = sym_from_upper(f64(s.G))
    info = torch.zeros(2, dtype=torch.int32, device=DEV)
    damp = torch.zeros(2, device=DEV)
    for pi_split in (False, True):
        info.zero_()
        kfac.kfac_damp_invert(step.invert_pairs(), GAMMA, pi_split=pi_split, info=info, damp=damp)
        torch.cuda.synchronize()
        assert info.cpu().tolist() == [0, 0], (case, pi_split)
        da, dg = oracle.pi_damping(A, G, GAMMA, pi_split)
        np.testing.assert_allclose(f64(damp), [da, dg], rtol=1e-4)
        for name, F, inv, dmp in (("A", A, s.A_inv, da), ("G", G, s.G_inv, dg)):
            X = f64(inv)
            R = F @ X + dmp * X - np.eye(F.shape[0])
            err = np.abs(R).max()
            assert err <= 1e-3, (case, name, "pi" if pi_split else "sqrt(gamma)", err)
        if pi_split:
            Ainv = oracle.damped_inverse(A, da)
            assert rel(f64(s.A_inv), Ainv) <= 1e-3, (case, rel(f64(s.A_inv), Ainv))
