"""GPU parity of the half-precision variant and of packed factor storage.

fp16 (Osawa et al. section 1: the factors are computed in half precision):
factor statistics from fp16 sources and the preconditioner with fp16
operands, against the oracle on the same fp16-rounded values, and an
accuracy / range comparison with bf16 on 1e-3-scale gradients.

Packed storage (section 1: the symmetry of the factors is exploited): the
factor update writing, and the inversion reading, the packed upper triangle
must give bitwise the results of the full row-major layout.
"""
import numpy as np
import pytest
import torch

import oracle
from second_order_optimisation_gb300 import kfac, workloads
from tests.test_gpu_parity import FACTOR_CASES

pytestmark = pytest.mark.gpu
DEV = "cuda"


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def word(ws):
    torch.cuda.synchronize()
    return int(ws[:4].view(torch.int32).item())


def _source(case, dtype, tag="f16"):
    name, shape, k, s, p, bias = case
    x = workloads.relu_normal_f32(shape, tag, name)
    xt = torch.from_numpy(x).to(dtype)
    xo = xt.float().numpy()
    xd = xt.to(DEV)
    if shape[1] == 1 and shape[2] == 1:
        xd = xd.reshape(shape[0], shape[3])
        xo = xo.reshape(shape[0], shape[3])
    P = oracle.im2col(xo, k, k, (s, s), (p, p), append_one=bias)
    return xd, P


# ------------------------------------------------------------- fp16 factors

@pytest.mark.parametrize("case", FACTOR_CASES, ids=[c[0] for c in FACTOR_CASES])
def test_factor_statistic_f16(case):
    """fp16 sources through every source path (direct rows, im2col tensor
    map, materialised patches, FC bias column): the raw statistic and the EMA
    from I against the oracle on the same fp16 values; fp16 products are
    exact in fp32, so the bound is the fp32 one."""
    _, _, k, s, p, bias = case
    xd, P = _source(case, torch.float16)
    M, d = P.shape
    S = oracle.gram(P)
    for xi in (0.0, 0.95):
        F = torch.eye(d, device=DEV) if xi else torch.zeros(d, d, device=DEV)
        ws = kfac.kfac_factor_update([kfac.FactorSource(xd, F, k, k, (s, s), (p, p), bias,
                                                        alpha=(1 - xi) / M, beta=xi)])
        assert word(ws) == 0
        ref = np.triu(xi * np.eye(d) + (1 - xi) * S / M)
        assert rel(np.triu(f64(F)), ref) <= 1e-4, (case[0], xi, rel(np.triu(f64(F)), ref))


def test_f16_vs_bf16_accuracy_and_range():
    """G from output gradients ~ N(0, 1e-3^2) given in fp32: fp16 keeps 3 more
    mantissa bits than bf16, so its statistic is closer to the oracle on the
    exact fp32 values; values beyond fp16's range (6.6e4) become infinite and
    the error word reports it, while bf16 (fp32's exponent range) keeps them;
    gradients of 1e-8 fall below fp16's smallest subnormal (6e-8) and are
    lost, while bf16 keeps them."""
    g = workloads.normal_f32((4096, 256), 1e-3, "f16cmp")
    S = oracle.gram(g.astype(np.float64)) / g.shape[0]
    errs = {}
    for dt in (torch.float16, torch.bfloat16):
        F = torch.zeros(256, 256, device=DEV)
        ws = kfac.kfac_factor_update([kfac.FactorSource(torch.from_numpy(g).to(dt).to(DEV), F,
                                                        alpha=1.0 / g.shape[0])])
        assert word(ws) == 0
        errs[dt] = rel(np.triu(f64(F)), np.triu(S))
    assert errs[torch.float16] < errs[torch.bfloat16] / 4, errs
    assert errs[torch.float16] <= 1e-3 and errs[torch.bfloat16] <= 2e-2, errs
    # range: activations of 1e5
    x = workloads.relu_normal_f32((512, 64), "f16big") * np.float32(1e5)
    for dt, finite in ((torch.float16, False), (torch.bfloat16, True)):
        F = torch.zeros(64, 64, device=DEV)
        ws = kfac.kfac_factor_update([kfac.FactorSource(torch.from_numpy(x).to(dt).to(DEV), F, alpha=1.0 / 512)])
        w = word(ws)
        assert bool(torch.isfinite(F).all()) == finite, dt
        assert bool(w & kfac.ERRW_NONFINITE) == (not finite), (dt, w)
    # underflow: gradients of 1e-8
    tiny = workloads.normal_f32((1024, 64), 1e-8, "f16tiny")
    St = oracle.gram(tiny.astype(np.float64)) / 1024
    out = {}
    for dt in (torch.float16, torch.bfloat16):
        F = torch.zeros(64, 64, device=DEV)
        kfac.kfac_factor_update([kfac.FactorSource(torch.from_numpy(tiny).to(dt).to(DEV), F, alpha=1.0 / 1024)])
        torch.cuda.synchronize()
        out[dt] = rel(np.triu(f64(F)), np.triu(St))
    assert out[torch.bfloat16] <= 2e-2 and out[torch.float16] > 0.5, out


# ------------------------------------------------------------- fp16 preconditioner

@pytest.mark.parametrize("dG,dA", [(32, 65), (130, 1001), (256, 576)])
def test_precondition_f16(dG, dA):
    """fp16 operands (the intermediate grad A^-1 rounded to fp16) against the
    oracle on the same fp16 values; fp16's error is below bf16's."""
    Gi = workloads.normal_f32((dG, dG), 1.0, "pc16", dG, dA, "G")
    Ai = workloads.normal_f32((dA, dA), 1.0, "pc16", dG, dA, "A")
    Gi, Ai = (Gi + Gi.T) / 2, (Ai + Ai.T) / 2
    grad = workloads.normal_f32((dG, dA), 1e-3, "pc16", dG, dA, "g")
    errs = {}
    for dt in (torch.float16, torch.bfloat16):
        host = [torch.from_numpy(a).to(dt) for a in (Gi, Ai, grad)]
        dev = []
        for h in host:
            r, c = h.shape
            buf = torch.zeros(r, (c + 7) // 8 * 8, dtype=dt, device=DEV)
            buf[:, :c] = h.to(DEV)
            dev.append(buf[:, :c])
        out = torch.empty(dG, dA, device=DEV)
        kfac.kfac_precondition([kfac.PrecondItem(dev[0], dev[1], dev[2], out)])
        torch.cuda.synchronize()
        Gh, Ah, gh = (h.float().numpy() for h in host)
        ref = oracle.precondition(Gh, gh, Ah)
        errs[dt] = rel(f64(out), ref)
    assert errs[torch.float16] <= 4e-3 and errs[torch.bfloat16] <= 2e-2, errs
    assert errs[torch.float16] < errs[torch.bfloat16], errs


def test_invert_f16_copies_are_the_rounded_inverse():
    A = torch.from_numpy(workloads.normal_f32((300, 300), 1.0, "inv16")).to(DEV)
    A = A @ A.T / 300
    G = torch.eye(70, device=DEV) * 2
    Ai, Gi = torch.empty_like(A), torch.empty_like(G)
    A16 = torch.empty(300, 304, dtype=torch.float16, device=DEV)[:, :300]
    G16 = torch.empty(70, 72, dtype=torch.float16, device=DEV)[:, :70]
    info = torch.zeros(2, dtype=torch.int32, device=DEV)
    kfac.kfac_damp_invert([kfac.InvertPair(A, G, Ai, Gi, A16, G16)], 1e-3, info=info)
    torch.cuda.synchronize()
    assert info.cpu().tolist() == [0, 0]
    assert torch.equal(A16, Ai.half()) and torch.equal(G16, Gi.half())


# ------------------------------------------------------------- packed storage

PACKED_CASES = [c for c in FACTOR_CASES if c[0] in ("fc_ragged", "fc_bias", "conv3x3", "conv7x7s2_c3",
                                                     "conv3x3s2_c128", "conv3x3_wide")]


@pytest.mark.parametrize("case", PACKED_CASES, ids=[c[0] for c in PACKED_CASES])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32], ids=["bf16", "f16", "f32"])
def test_factor_packed_equals_full(case, dtype):
    """The packed upper triangle the update writes is bitwise the upper
    triangle of the full-layout update (raw statistic and EMA over two calls),
    and matches the oracle."""
    _, _, k, s, p, bias = case
    xd, P = _source(case, dtype, "packed")
    M, d = P.shape
    F = torch.eye(d, device=DEV)
    Fp = kfac.pack_upper(torch.eye(d, device=DEV))
    for call in range(2):
        for dst, packed in ((F, False), (Fp, True)):
            ws = kfac.kfac_factor_update([kfac.FactorSource(xd, dst, k, k, (s, s), (p, p), bias,
                                                            alpha=0.05 / M, beta=0.95, packed=packed)])
            assert word(ws) == 0
    torch.cuda.synchronize()
    assert torch.equal(Fp, kfac.pack_upper(F))
    ref = oracle.factor_ema(oracle.factor_ema(np.eye(d), P, 0.95), P, 0.95)
    tol = 1e-4 if dtype != torch.bfloat16 else 2e-2
    assert rel(oracle.unpack_upper(f64(Fp), d), ref) <= tol


def test_invert_packed_equals_full():
    """Damped inversion reading packed factors gives bitwise the inverses and
    damping of the full layout, for several sizes in one call."""
    dims = [(300, 130), (64, 257), (1024, 40)]
    pairs_f, pairs_p, outs = [], [], []
    for da, dg in dims:
        Xa = torch.from_numpy(workloads.normal_f32((2 * da, da), 1.0, "pk", da)).to(DEV)
        Xg = torch.from_numpy(workloads.normal_f32((2 * dg, dg), 1.0, "pk", dg)).to(DEV)
        A = Xa.T @ Xa / (2 * da)
        G = Xg.T @ Xg / (2 * dg)
        of = [torch.empty(da, da, device=DEV), torch.empty(dg, dg, device=DEV)]
        op = [torch.empty(da, da, device=DEV), torch.empty(dg, dg, device=DEV)]
        pairs_f.append(kfac.InvertPair(A, G, *of))
        pairs_p.append(kfac.InvertPair(kfac.pack_upper(A), kfac.pack_upper(G), *op, dA=da, dG=dg,
                                       packed_A=True, packed_G=True))
        outs.append((of, op))
    df = torch.zeros(2 * len(dims), device=DEV)
    dp = torch.zeros(2 * len(dims), device=DEV)
    info = torch.zeros(2 * len(dims), dtype=torch.int32, device=DEV)
    kfac.kfac_damp_invert(pairs_f, 1e-3, damp=df)
    kfac.kfac_damp_invert(pairs_p, 1e-3, damp=dp, info=info)
    torch.cuda.synchronize()
    assert int(info.abs().sum().item()) == 0
    assert torch.equal(df, dp)
    for of, op in outs:
        assert torch.equal(of[0], op[0]) and torch.equal(of[1], op[1])
