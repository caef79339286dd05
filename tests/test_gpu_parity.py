"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs, at sizes the oracle finishes in seconds that still
span several 128-wide tiles and a ragged tail.

Tolerances (relative Frobenius error unless stated):
  factors / preconditioned gradients from bf16 inputs   <= 2e-2
  factors / preconditioned gradients from fp32 inputs   <= 1e-4
  damped inverses: max |(F + damp I) inv - I|           <= 1e-3
"""
import numpy as np
import pytest
import torch

import oracle
from second_order_optimisation_gb300 import kfac, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def bf16(a):
    return workloads.to_bf16(a)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


# -------------------------------------------------------------- BN diag Fisher

@pytest.mark.parametrize("C,ns", [(64, 1024), (96, 33), (7, 5), (2048, 1024), (130, 17)])
def test_bn_diag_fisher(C, ns):
    x = workloads.normal_f32((ns, C), 1e-2, "bn", C, ns)
    xd = torch.from_numpy(x).to(DEV)
    F = torch.full((C,), 0.5, device=DEV)
    g = torch.empty(C, device=DEV)
    p = torch.empty(C, device=DEV)
    kfac.kfac_bn_diag_fisher([kfac.BnItem(xd, F, p, g)], 1e-3, xi=0.0)
    torch.cuda.synchronize()
    Fo, go, po = oracle.bn_diag_fisher(x, 1e-3)
    assert rel(f64(F), Fo) <= 1e-4
    assert rel(f64(g), go) <= 1e-4
    assert rel(f64(p), po) <= 1e-4


def test_bn_diag_fisher_ema_and_many_layers():
    chans = [64, 256, 33, 2048, 512]
    items, ref = [], []
    for i, C in enumerate(chans):
        x = workloads.normal_f32((64, C), 1e-2, "bnmany", i)
        F0 = np.full(C, 0.25, dtype=np.float32)
        it = kfac.BnItem(torch.from_numpy(x).to(DEV), torch.from_numpy(F0).to(DEV),
                         torch.empty(C, device=DEV), torch.empty(C, device=DEV))
        items.append(it)
        ref.append(oracle.bn_diag_fisher(x, 1e-3, xi=0.9, F=F0))
    kfac.kfac_bn_diag_fisher(items, 1e-3, xi=0.9)
    torch.cuda.synchronize()
    for it, (Fo, go, po) in zip(items, ref):
        assert rel(f64(it.F), Fo) <= 1e-4
        assert rel(f64(it.precond), po) <= 1e-4


# -------------------------------------------------------------- factor update

FACTOR_CASES = [
    # name, (n, h, w, c), k, stride, pad, append_one
    ("fc_ragged", (300, 1, 1, 200), 1, 1, 0, False),
    ("fc_bias", (77, 1, 1, 136), 1, 1, 0, True),
    ("fc_small_d", (1000, 1, 1, 8), 1, 1, 0, False),
    ("conv3x3", (3, 9, 9, 64), 3, 1, 1, False),
    ("conv7x7s2_c3", (2, 15, 15, 3), 7, 2, 3, False),
    ("conv1x1s2", (2, 10, 10, 72), 1, 2, 0, False),
    ("conv1x1_tall", (16, 14, 14, 64), 1, 1, 0, False),
    ("conv3x3_wide", (2, 7, 7, 136), 3, 1, 1, False),
    # channels in whole 64-wide taps: bf16 reads the input through an im2col tensor map
    ("conv3x3s2_c128", (3, 11, 11, 128), 3, 2, 1, False),
    ("conv1x1s2_c64", (2, 9, 9, 64), 1, 2, 0, False),
    ("conv3x3_c192_wrap", (5, 5, 5, 192), 3, 1, 1, False),
]


@pytest.mark.parametrize("case", FACTOR_CASES, ids=[c[0] for c in FACTOR_CASES])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_factor_statistic(case, dtype):
    """Raw statistic (beta = 0, alpha = 1/M) and the EMA form from I, upper
    triangle only; entries below the diagonal must stay untouched."""
    name, shape, k, s, p, bias = case
    x = workloads.relu_normal_f32(shape, "factor", name)
    if dtype == "bf16":
        xt = bf16(x)
        xo = xt.float().numpy()
    else:
        xt = torch.from_numpy(x)
        xo = x
    xd = xt.to(DEV)
    if shape[1] == 1 and shape[2] == 1:
        xd = xd.reshape(shape[0], shape[3])
        xo2 = xo.reshape(shape[0], shape[3])
    else:
        xo2 = xo
    P = oracle.im2col(xo2, k, k, (s, s), (p, p), append_one=bias)
    M, d = P.shape
    S = oracle.gram(P)
    ldf = d + 5
    sentinel = -12345.0
    for xi in (0.0, 0.95):
        F = torch.full((d, ldf), sentinel, device=DEV)
        up_mask = torch.triu(torch.ones(d, d, dtype=torch.bool, device=DEV))
        init = torch.eye(d, device=DEV) if xi else torch.zeros(d, d, device=DEV)
        F[:, :d] = torch.where(up_mask, init, torch.full_like(init, sentinel))
        src = kfac.FactorSource(xd, F, k, k, (s, s), (p, p), bias, alpha=(1 - xi) / M, beta=xi)
        ws = kfac.kfac_factor_update([src])
        torch.cuda.synchronize()
        assert int(ws[:4].view(torch.int32).item()) == 0
        Fh = F.cpu().numpy().astype(np.float64)
        up = np.triu(Fh[:, :d])
        ref = np.triu(xi * np.eye(d) + (1 - xi) * S / M)
        tol = 2e-2 if dtype == "bf16" else 1e-4
        assert rel(up, ref) <= tol, (xi, rel(up, ref))
        low = np.tril(np.ones((d, d), bool), -1)
        assert np.all(Fh[:, :d][low] == sentinel)   # strictly-lower entries never written
        assert np.all(Fh[:, d:] == sentinel)        # nothing written past d


def test_factor_many_layers_one_call():
    """A heterogeneous batch (several layers, A and G) in one call."""
    layers = [workloads.Layer("a", 64, 40, 3, 1, 1, 6, 6), workloads.Layer("b", 24, 136, 1, 2, 0, 8, 4),
              workloads.Layer("c", 136, 256, 1, 1, 0, 5, 5)]
    srcs, refs = [], []
    for L in layers:
        x, g, _ = workloads.layer_inputs(L, 3, "many", grad_w=False)
        M = L.rows(3)
        A = torch.zeros(L.d_a, L.d_a, device=DEV)
        G = torch.zeros(L.d_g, L.d_g, device=DEV)
        srcs.append(kfac.FactorSource(x.to(DEV), A, L.k, L.k, (L.stride,) * 2, (L.pad,) * 2,
                                      alpha=1.0 / M))
        srcs.append(kfac.FactorSource(g.to(DEV), G, alpha=1.0 / M))
        P = oracle.im2col(x.float().numpy(), L.k, L.k, (L.stride,) * 2, (L.pad,) * 2)
        refs.append(oracle.gram(P) / M)
        refs.append(oracle.gram(g.float().numpy()) / M)
    kfac.kfac_factor_update(srcs)
    torch.cuda.synchronize()
    for s_, r in zip(srcs, refs):
        assert rel(np.triu(f64(s_.F)), np.triu(r)) <= 2e-2


def test_factor_repeated_batched_calls_and_workspace_bounds():
    """The same heterogeneous batch (im2col and direct sources) three times in
    a row with beta = 0 gives the same, correct statistics each time, and
    nothing is written past the workspace size the library asks for."""
    layers = [workloads.Layer("c7", 3, 16, 7, 2, 3, 18, 9), workloads.Layer("c3", 64, 72, 3, 1, 1, 6, 6),
              workloads.Layer("c1", 136, 64, 1, 1, 0, 5, 5)]
    srcs, refs = [], []
    for L in layers:
        x, g, _ = workloads.layer_inputs(L, 4, "repeat", grad_w=False)
        M = L.rows(4)
        srcs.append(kfac.FactorSource(x.to(DEV), torch.zeros(L.d_a, L.d_a, device=DEV), L.k, L.k,
                                      (L.stride,) * 2, (L.pad,) * 2, alpha=1.0 / M))
        srcs.append(kfac.FactorSource(g.to(DEV), torch.zeros(L.d_g, L.d_g, device=DEV), alpha=1.0 / M))
        P = oracle.im2col(x.float().numpy(), L.k, L.k, (L.stride,) * 2, (L.pad,) * 2)
        refs += [oracle.gram(P) / M, oracle.gram(g.float().numpy()) / M]
    need = kfac.kfac_factor_update_workspace_size(srcs)
    ws = torch.full((need + 4096,), 0xAB, dtype=torch.uint8, device=DEV)
    first = None
    for call in range(3):
        kfac.kfac_factor_update(srcs, ws[:need])
        torch.cuda.synchronize()
        got = [np.triu(f64(s_.F)) for s_ in srcs]
        for gt, r in zip(got, refs):
            assert np.all(np.isfinite(gt)) and rel(gt, np.triu(r)) <= 2e-2
        if first is None:
            first = got
        else:
            for a_, b_ in zip(got, first):
                assert np.array_equal(a_, b_)        # deterministic across calls
    assert int((ws[need:] != 0xAB).sum().item()) == 0


def test_factor_chunked_accumulation():
    """Statistic accumulated over 4 chunks (beta = xi, then 1) equals the
    single statistic of all rows (gradient accumulation, section 2)."""
    x = bf16(workloads.relu_normal_f32((4 * 50, 96), "chunks"))
    M, xi = 200, 0.95
    Fa = torch.eye(96, device=DEV)
    for c in range(4):
        kfac.kfac_factor_update([kfac.FactorSource(x[c * 50:(c + 1) * 50].contiguous().to(DEV), Fa,
                                                   alpha=(1 - xi) / M, beta=xi if c == 0 else 1.0)])
    torch.cuda.synchronize()
    ref = oracle.factor_ema(np.eye(96), x.float().numpy(), xi)
    assert rel(np.triu(f64(Fa)), np.triu(ref)) <= 2e-2


# -------------------------------------------------------------- damped inverse

def _spd_factor(d, tag, M=None, xi=0.0):
    M = M or max(2 * d, 16)
    P = workloads.relu_normal_f32((M, d), "inv", tag)
    return oracle.factor_ema(np.eye(d), P, xi) if xi else oracle.gram(P) / M


@pytest.mark.parametrize("dA,dG", [(1, 1), (5, 3), (64, 128), (129, 127), (200, 64), (300, 257),
                                   (700, 130), (2049, 1000)])
def test_damp_invert(dA, dG):
    A = _spd_factor(dA, f"A{dA}").astype(np.float32)
    G = (_spd_factor(dG, f"G{dG}") * 1e-4).astype(np.float32)
    gamma = 1e-3
    Ad = torch.from_numpy(np.triu(A)).to(DEV)       # only the upper triangle is read
    Gd = torch.from_numpy(np.triu(G)).to(DEV)
    Ai = torch.empty(dA, dA, device=DEV)
    Gi = torch.empty(dG, dG + 3, device=DEV)
    lda16 = (dA + 7) // 8 * 8
    Ab = torch.empty(dA, lda16, dtype=torch.bfloat16, device=DEV)
    info = torch.full((2,), -7, dtype=torch.int32, device=DEV)
    damp = torch.empty(2, device=DEV)
    kfac.kfac_damp_invert([kfac.InvertPair(Ad, Gd, Ai, Gi[:, :dG], Ab[:, :dA], None)], gamma,
                          info=info, damp=damp)
    torch.cuda.synchronize()
    assert info.cpu().tolist() == [0, 0]
    da, dg = oracle.pi_damping(A.astype(np.float64), G.astype(np.float64), gamma)
    np.testing.assert_allclose(damp.cpu().numpy(), [da, dg], rtol=1e-4)
    for F, inv, dmp in ((A, f64(Ai), da), (G, f64(Gi[:, :dG]), dg)):
        d = F.shape[0]
        R = (F.astype(np.float64) + dmp * np.eye(d)) @ inv - np.eye(d)
        assert np.abs(R).max() <= 1e-3, np.abs(R).max()
        assert np.array_equal(inv, inv.T)
        ref = oracle.damped_inverse(F.astype(np.float64), dmp)
        assert rel(inv, ref) <= 1e-3
    np.testing.assert_allclose(f64(Ab[:, :dA]), f64(Ai), rtol=1e-2, atol=1e-2 * np.abs(f64(Ai)).max())


def test_damp_invert_two_groups_eager_and_graph():
    """Chains of very different length (1024- and 640-wide factors next to
    200- and 64-wide ones) run as two concurrent groups on library streams.
    Eager and graph-captured calls agree bitwise, and every inverse meets the
    residual bound."""
    dims = [(1024, 200), (640, 64), (200, 130)]
    gamma = 1e-3
    pairs, host = [], []
    for dA, dG in dims:
        A = _spd_factor(dA, f"A{dA}g").astype(np.float32)
        G = (_spd_factor(dG, f"G{dG}g") * 1e-3).astype(np.float32)
        host.append((A, G))
        pairs.append(kfac.InvertPair(torch.from_numpy(np.triu(A)).to(DEV), torch.from_numpy(np.triu(G)).to(DEV),
                                     torch.empty(dA, dA, device=DEV), torch.empty(dG, dG, device=DEV)))
    ws = torch.empty(kfac.kfac_damp_invert_workspace_size(pairs), dtype=torch.uint8, device=DEV)
    info = torch.full((2 * len(dims),), -7, dtype=torch.int32, device=DEV)
    damp = torch.empty(2 * len(dims), device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kfac.kfac_damp_invert(pairs, gamma, info=info, damp=damp, workspace=ws, stream=s)
    torch.cuda.synchronize()
    assert info.cpu().tolist() == [0] * (2 * len(dims))
    assert int(ws[:4].view(torch.int32).item()) == 0  # device error word: no wait ran out
    eager = [(f64(p.A_inv), f64(p.G_inv)) for p in pairs]
    for p in pairs:
        p.A_inv.zero_()
        p.G_inv.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kfac.kfac_damp_invert(pairs, gamma, info=info, damp=damp, workspace=ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    dm = damp.cpu().numpy().astype(np.float64)
    for l, ((A, G), p, (ea, eg)) in enumerate(zip(host, pairs, eager)):
        ga, gg = f64(p.A_inv), f64(p.G_inv)
        assert np.array_equal(ga, ea) and np.array_equal(gg, eg)
        for F, inv, dmp in ((A, ga, dm[2 * l]), (G, gg, dm[2 * l + 1])):
            R = (F.astype(np.float64) + dmp * np.eye(F.shape[0])) @ inv - np.eye(F.shape[0])
            assert np.abs(R).max() <= 1e-3, np.abs(R).max()


def test_damp_invert_not_pd_reports_info():
    """-I with gamma = 0 and no pi split: the first pivot fails; info says so
    and nothing hangs."""
    for d in (5, 200):
        A = torch.triu(-torch.eye(d, device=DEV))
        G = torch.eye(3, device=DEV)
        info = torch.zeros(2, dtype=torch.int32, device=DEV)
        kfac.kfac_damp_invert([kfac.InvertPair(A, G, torch.empty_like(A), torch.empty_like(G))], 0.0,
                              pi_split=False, info=info)
        torch.cuda.synchronize()
        assert info.cpu().tolist() == [1, 0]


@pytest.mark.parametrize("d,bad", [(200, 77), (200, 199), (256, 255), (600, 450), (600, 130)])
def test_damp_invert_not_pd_deep_pivot(d, bad):
    """A positive diagonal with one negative entry (gamma = 0, no pi split):
    the first failing pivot is that entry, inside a later 32-wide block step
    of a 256-row leaf or in a later leaf of the recursion; info gives its
    1-based index and every other pivot still eliminates normally."""
    diag = torch.linspace(1.0, 2.0, d, device=DEV)
    diag[bad] = -0.5
    A = torch.diag(diag)
    G = torch.eye(3, device=DEV)
    Ai = torch.empty_like(A)
    info = torch.zeros(2, dtype=torch.int32, device=DEV)
    kfac.kfac_damp_invert([kfac.InvertPair(A, G, Ai, torch.empty_like(G))], 0.0, pi_split=False, info=info)
    torch.cuda.synchronize()
    assert info.cpu().tolist() == [bad + 1, 0]
    # the other diagonal entries are still inverted (a diagonal matrix has no coupling)
    ok = torch.ones(d, dtype=torch.bool)
    ok[bad] = False
    got = torch.diagonal(Ai).cpu()[ok].double()
    np.testing.assert_allclose(got.numpy(), (1.0 / diag.cpu()[ok].double()).numpy(), rtol=1e-5)


# -------------------------------------------------------------- precondition

@pytest.mark.parametrize("dG,dA", [(32, 65), (128, 200), (256, 576), (130, 1001)])
def test_precondition_bf16(dG, dA):
    rng_tag = ("pc", dG, dA)
    Gi = workloads.normal_f32((dG, dG), 1.0, *rng_tag, "G")
    Gi = (Gi + Gi.T) / 2
    Ai = workloads.normal_f32((dA, dA), 1.0, *rng_tag, "A")
    Ai = (Ai + Ai.T) / 2
    grad = workloads.normal_f32((dG, dA), 1e-3, *rng_tag, "g")
    Gb, Ab, gb = bf16(Gi), bf16(Ai), bf16(grad)
    ld = (dA + 7) // 8 * 8
    Abd = torch.zeros(dA, ld, dtype=torch.bfloat16, device=DEV)
    Abd[:, :dA] = Ab.to(DEV)
    gd = torch.zeros(dG, ld, dtype=torch.bfloat16, device=DEV)
    gd[:, :dA] = gb.to(DEV)
    ldg = (dG + 7) // 8 * 8
    Gd = torch.zeros(dG, ldg, dtype=torch.bfloat16, device=DEV)
    Gd[:, :dG] = Gb.to(DEV)
    out = torch.empty(dG, dA, device=DEV)
    kfac.kfac_precondition([kfac.PrecondItem(Gd[:, :dG], Abd[:, :dA], gd[:, :dA], out)])
    torch.cuda.synchronize()
    ref = oracle.precondition(Gb.float().numpy(), gb.float().numpy(), Ab.float().numpy())
    assert rel(f64(out), ref) <= 2e-2


def test_precondition_f32():
    dG, dA = 70, 133
    Gi = workloads.normal_f32((dG, dG), 1.0, "pcf", "G")
    Ai = workloads.normal_f32((dA, dA), 1.0, "pcf", "A")
    grad = workloads.normal_f32((dG, dA), 1e-3, "pcf", "g")
    out = torch.empty(dG, dA, device=DEV)
    kfac.kfac_precondition([kfac.PrecondItem(torch.from_numpy(Gi).to(DEV), torch.from_numpy(Ai).to(DEV),
                                             torch.from_numpy(grad).to(DEV), out)])
    torch.cuda.synchronize()
    assert rel(f64(out), oracle.precondition(Gi, grad, Ai)) <= 1e-4


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_precondition_clears_error_word(dtype):
    """The first int32 of the workspace is the device error word: every call
    sets it to 0 before its kernels, whatever the operand dtype."""
    dG, dA = 40, 72
    G = torch.eye(dG, device=DEV, dtype=dtype)
    A = torch.eye(dA, device=DEV, dtype=dtype)
    g = torch.ones(dG, dA, device=DEV, dtype=dtype)
    out = torch.empty(dG, dA, device=DEV)
    items = [kfac.PrecondItem(G, A, g, out)]
    ws = torch.zeros(kfac.kfac_precondition_workspace_size(items), dtype=torch.uint8, device=DEV)
    ws[:4].view(torch.int32).fill_(-1)
    kfac.kfac_precondition(items, ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    assert bool((out == 1.0).all())


# -------------------------------------------------------------- fused step on the weights (Eq. 8)

def _precond_operands(dG, dA, dtype, tag):
    """Symmetric inverses and a 1e-3-scale gradient; bf16 operands sit in
    row-padded buffers (ld a multiple of 8) so the views have ragged widths."""
    Gi = workloads.normal_f32((dG, dG), 1.0, "wu", tag, "G")
    Ai = workloads.normal_f32((dA, dA), 1.0, "wu", tag, "A")
    Gi, Ai = (Gi + Gi.T) / 2, (Ai + Ai.T) / 2
    grad = workloads.normal_f32((dG, dA), 1e-3, "wu", tag, "g")
    if dtype == torch.float32:
        return ([torch.from_numpy(x).to(DEV) for x in (Gi, Ai, grad)], (Gi, Ai, grad))
    host = [bf16(x) for x in (Gi, Ai, grad)]
    dev = []
    for x in host:
        r, c = x.shape
        buf = torch.zeros(r, (c + 7) // 8 * 8, dtype=torch.bfloat16, device=DEV)
        buf[:, :c] = x.to(DEV)
        dev.append(buf[:, :c])
    return dev, tuple(x.float().numpy() for x in host)


@pytest.mark.parametrize("dtype,dG,dA", [(torch.bfloat16, 130, 1001), (torch.bfloat16, 256, 576),
                                         (torch.float32, 70, 133), (torch.float32, 129, 260)],
                         ids=["bf16-130x1001", "bf16-256x576", "fp32-70x133", "fp32-129x260"])
@pytest.mark.parametrize("keep_out", [True, False], ids=["out", "no-out"])
def test_precondition_fused_weight_update(dtype, dG, dA, keep_out):
    """w <- w - eta * (G^-1 grad A^-1) in the second product's epilogue, against
    the oracle's preconditioned gradient and update; with out kept, out is
    bitwise the unfused result and w is one fused multiply-add of it."""
    (Gd, Ad, gd), (Gh, Ah, gh) = _precond_operands(dG, dA, dtype, f"{dtype}{dG}x{dA}")
    eta = 0.125
    w0 = workloads.normal_f32((dG, dA), 5e-2, "wu", dG, dA, "w")
    ldw = dA + 3  # padded rows (16-byte row access only where dA + 3 is a multiple of 4)
    wbuf = torch.zeros(dG, ldw, device=DEV)
    wbuf[:, :dA] = torch.from_numpy(w0).to(DEV)
    w = wbuf[:, :dA]
    out = torch.empty(dG, dA, device=DEV) if keep_out else None
    kfac.kfac_precondition([kfac.PrecondItem(Gd, Ad, gd, out, w=w, eta=eta)])
    plain = torch.empty(dG, dA, device=DEV)
    kfac.kfac_precondition([kfac.PrecondItem(Gd, Ad, gd, plain)])
    torch.cuda.synchronize()
    P_ref = oracle.precondition(Gh, gh, Ah)
    w_ref = oracle.weight_update(w0.astype(np.float64), P_ref, eta)
    tol = 2e-2 if dtype == torch.bfloat16 else 1e-4
    assert rel(f64(w) - w0, w_ref - w0) <= tol
    assert rel(f64(w), w_ref) <= tol
    assert bool((wbuf[:, dA:] == 0).all())  # the row padding is untouched
    if keep_out:
        assert torch.equal(out, plain)
    np.testing.assert_allclose(f64(w), w0.astype(np.float64) - np.float64(np.float32(eta)) * f64(plain),
                               rtol=3e-7, atol=1e-9)


def test_precondition_weight_update_only_rejects_no_destination():
    G = torch.eye(8, device=DEV)
    g = torch.ones(8, 8, device=DEV)
    with pytest.raises(kfac.KfacError):
        kfac.kfac_precondition([kfac.PrecondItem(G, G, g, None)])


# -------------------------------------------------------------- whole layer step

def test_fc64x32_fp32_step():
    """The single-FC-layer case: a[32,64] + bias column, g[32,32], fp32,
    factors from I, xi = 0.95, gamma = 1e-3 split by pi."""
    a, g = workloads.fc_small_fp32()
    P = oracle.im2col(a.astype(np.float64), append_one=True)
    grad = oracle.weight_grad(P, g.astype(np.float64), 32)
    ref = oracle.kfac_layer_step(np.eye(65), np.eye(32), P, g.astype(np.float64), grad, xi=0.95,
                                 gamma=1e-3)
    A = torch.eye(65, device=DEV)
    G = torch.eye(32, device=DEV)
    kfac.kfac_factor_update([kfac.FactorSource(torch.from_numpy(a).to(DEV), A, append_one=True,
                                               alpha=0.05 / 32, beta=0.95),
                             kfac.FactorSource(torch.from_numpy(g).to(DEV), G, alpha=0.05 / 32, beta=0.95)])
    Ai, Gi = torch.empty_like(A), torch.empty_like(G)
    info = torch.zeros(2, dtype=torch.int32, device=DEV)
    kfac.kfac_damp_invert([kfac.InvertPair(A, G, Ai, Gi)], 1e-3, info=info)
    out = torch.empty(32, 65, device=DEV)
    kfac.kfac_precondition([kfac.PrecondItem(Gi, Ai, torch.from_numpy(grad.astype(np.float32)).to(DEV), out)])
    torch.cuda.synchronize()
    assert info.cpu().tolist() == [0, 0]
    assert rel(np.triu(f64(A)), np.triu(ref["A"])) <= 1e-4
    assert rel(np.triu(f64(G)), np.triu(ref["G"])) <= 1e-4
    for F, inv, dmp in ((ref["A"], f64(Ai), ref["damp_A"]), (ref["G"], f64(Gi), ref["damp_G"])):
        R = (F + dmp * np.eye(F.shape[0])) @ inv - np.eye(F.shape[0])
        assert np.abs(R).max() <= 1e-3
    assert rel(f64(out), ref["precond"]) <= 1e-4


def test_timing_records_every_launch():
    """The diagnostic per-launch record: one entry per library launch, in
    enqueue order, with its kernel kind; reading clears it."""
    x = bf16(workloads.relu_normal_f32((2, 9, 9, 64), "timing")).to(DEV)
    F = torch.zeros(576, 576, device=DEV)
    kfac.timing_enable(True)
    kfac.timing_read_launches()
    n0 = kfac.launch_count()
    kfac.kfac_factor_update([kfac.FactorSource(x, F, 3, 3, (1, 1), (1, 1), alpha=1.0 / 162)])
    n1 = kfac.launch_count()
    rec = kfac.timing_read_launches()
    kfac.timing_enable(False)
    assert len(rec) == n1 - n0 > 0
    assert all(d >= 0.0 for _, d, _, _ in rec) and rec[0][0] == 0.0
    assert "tc_gemm_bf16" in {k for _, _, k, _ in rec}
    assert {sid for _, _, _, sid in rec} == {0}  # all on the caller's stream
    assert kfac.timing_read_launches() == []
