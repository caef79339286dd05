"""Error paths on the GPU: NaN / infinite data in a factor source, a factor
or a gradient, and fp32 overflow of the statistic or of the updated weights.

Each call's device error word (the first int32 of its workspace) must carry
ERRW_NONFINITE after such data and be 0 after a clean call; the damped
inversion must report the failing factor in info (a pivot that is not
positive and finite); and the other layers of the same batched call must come
out exactly as in a clean call of the same shapes (the failure stays in its
layer).  The data are ordinary values (NaN, inf, 1e20): nothing here makes a
kernel wait, trap or touch memory out of bounds.
"""
import math

import pytest
import torch

from second_order_optimisation_gb300 import kfac, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def word(ws):
    torch.cuda.synchronize()
    return int(ws[:4].view(torch.int32).item())


def bf16_dev(a):
    return workloads.to_bf16(a).to(DEV)


# ------------------------------------------------------------- factor statistic

def _factor_call(x0, g1):
    """Two factor updates in one call: A0 from NHWC x0 (3x3 taps), G1 from
    rows g1; returns (F0, F1, error word)."""
    F0 = torch.eye(9 * x0.shape[-1], device=DEV)
    F1 = torch.eye(g1.shape[1], device=DEV)
    srcs = [kfac.FactorSource(x0, F0, 3, 3, (1, 1), (1, 1), alpha=0.05 / 200, beta=0.95),
            kfac.FactorSource(g1, F1, alpha=0.05 / 200, beta=0.95)]
    ws = kfac.kfac_factor_update(srcs)
    return F0, F1, word(ws)


@pytest.mark.parametrize("bad", [math.nan, math.inf, -math.inf], ids=["nan", "inf", "-inf"])
def test_factor_nonfinite_source_sets_word_and_stays_in_its_layer(bad):
    x = workloads.relu_normal_f32((2, 10, 10, 64), "err-x")
    g = workloads.normal_f32((200, 96), 1e-3, "err-g")
    F0c, F1c, wc = _factor_call(bf16_dev(x), bf16_dev(g))
    assert wc == 0
    xb = x.copy()
    xb[1, 4, 7, 33] = bad
    F0, F1, w = _factor_call(bf16_dev(xb), bf16_dev(g))
    assert w & kfac.ERRW_NONFINITE
    assert not bool(torch.isfinite(F0).all())
    assert torch.equal(F1, F1c)            # the other layer of the call is untouched
    # the entries whose patches never see the bad pixel are still finite
    assert bool(torch.isfinite(F0[0, :]).any())


def test_factor_fp32_source_inf_and_overflow():
    """fp32 sources take the CUDA-core path: an infinite value, and finite
    values whose squares overflow fp32 (1e20^2), both set the bit."""
    rows = torch.from_numpy(workloads.normal_f32((64, 40), 1.0, "err-f32")).to(DEV)
    for poison in (math.inf, 1e20):
        r = rows.clone()
        r[5, 3] = poison
        F = torch.zeros(40, 40, device=DEV)
        ws = kfac.kfac_factor_update([kfac.FactorSource(r, F, alpha=1.0, beta=0.0)])
        assert word(ws) & kfac.ERRW_NONFINITE, poison
    F = torch.zeros(40, 40, device=DEV)
    ws = kfac.kfac_factor_update([kfac.FactorSource(rows, F, alpha=1.0, beta=0.0)])
    assert word(ws) == 0


def test_factor_bf16_statistic_overflow():
    """Finite bf16 inputs of 1e20: the fp32 statistic overflows to inf."""
    g = workloads.normal_f32((256, 128), 1e-3, "err-ovf")
    g[17, :] = 1e20
    F = torch.zeros(128, 128, device=DEV)
    ws = kfac.kfac_factor_update([kfac.FactorSource(bf16_dev(g), F, alpha=1.0, beta=0.0)])
    assert word(ws) & kfac.ERRW_NONFINITE
    assert bool(torch.isinf(F).any())


# ------------------------------------------------------------- damped inversion

def _spd(d, tag):
    X = workloads.normal_f32((4 * d, d), 1.0, "err-spd", tag, d)
    X = torch.from_numpy(X).double()
    return ((X.T @ X) / (4 * d)).float().to(DEV)


@pytest.mark.parametrize("where", ["offdiag-nan", "diag-inf", "corner-nan"])
def test_invert_nonfinite_factor_reports_info_and_word(where):
    dA0, dG0, dA1, dG1 = 300, 130, 257, 64
    A0, G0, A1, G1 = _spd(dA0, "a0"), _spd(dG0, "g0"), _spd(dA1, "a1"), _spd(dG1, "g1")

    def call(A0x):
        outs = [torch.empty_like(m) for m in (A0x, G0, A1, G1)]
        info = torch.full((4,), -7, dtype=torch.int32, device=DEV)
        ws = kfac.kfac_damp_invert([kfac.InvertPair(A0x, G0, outs[0], outs[1]),
                                    kfac.InvertPair(A1, G1, outs[2], outs[3])], 1e-3, info=info)
        return outs, info.cpu().tolist(), word(ws)

    clean, info_c, wc = call(A0)
    assert info_c == [0, 0, 0, 0] and wc == 0
    Ab = A0.clone()
    if where == "offdiag-nan":
        Ab[100, 250] = math.nan          # upper triangle: read
    elif where == "diag-inf":
        Ab[200, 200] = math.inf
    else:
        Ab[dA0 - 1, dA0 - 1] = math.nan  # the very last pivot
    outs, info, w = call(Ab)
    assert info[0] > 0, info             # 1-based index of the first failing pivot
    assert info[1:] == [0, 0, 0]
    assert w & kfac.ERRW_NONFINITE
    for k in (2, 3):                     # the other layer: as in the clean call
        assert torch.equal(outs[k], clean[k]), k
    # G of the same layer stays a finite inverse; a NaN or infinite diagonal
    # entry of A leaves its trace (and so the pi split) undefined, and both
    # factors fall back to sqrt(gamma): G's values may then differ from the
    # clean call's
    assert bool(torch.isfinite(outs[1]).all())
    if where == "offdiag-nan":
        assert torch.equal(outs[1], clean[1])


def test_invert_nan_in_lower_triangle_is_ignored():
    """Only the upper triangle of a factor is read: NaN below the diagonal
    changes nothing."""
    A = _spd(200, "low")
    G = _spd(72, "lowg")
    outs0 = [torch.empty_like(A), torch.empty_like(G)]
    kfac.kfac_damp_invert([kfac.InvertPair(A, G, *outs0)], 1e-3)
    Ab = A.clone()
    Ab[150, 20] = math.nan
    outs1 = [torch.empty_like(A), torch.empty_like(G)]
    info = torch.zeros(2, dtype=torch.int32, device=DEV)
    ws = kfac.kfac_damp_invert([kfac.InvertPair(Ab, G, *outs1)], 1e-3, info=info)
    assert word(ws) == 0
    assert info.cpu().tolist() == [0, 0]
    assert torch.equal(outs0[0], outs1[0]) and torch.equal(outs0[1], outs1[1])


# ------------------------------------------------------------- preconditioner

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_precondition_nonfinite_gradient(dtype):
    shapes = [(96, 200), (64, 136)]
    items, outs = [], []
    for k, (dG, dA) in enumerate(shapes):
        G = torch.eye(dG, device=DEV, dtype=dtype) * 2
        A = torch.eye(dA, device=DEV, dtype=dtype) * 0.5
        g = torch.from_numpy(workloads.normal_f32((dG, dA), 1e-3, "err-pc", k)).to(DEV, dtype)
        items.append([G, A, g])
    def call(poison):
        res = []
        its = []
        for k, (G, A, g) in enumerate(items):
            gg = g.clone()
            if k == 0 and poison is not None:
                gg[10, 20] = poison
            o = torch.empty(gg.shape, device=DEV)
            res.append(o)
            its.append(kfac.PrecondItem(G, A, gg, o))
        ws = kfac.kfac_precondition(its)
        return res, word(ws)
    clean, wc = call(None)
    assert wc == 0
    for poison in (math.nan, math.inf):
        res, w = call(poison)
        assert w & kfac.ERRW_NONFINITE
        assert not bool(torch.isfinite(res[0]).all())
        assert torch.equal(res[1], clean[1])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_weight_update_overflow(dtype):
    """w near the fp32 maximum pushed past it by -eta * P: the updated weight
    is infinite and the word says so."""
    dG, dA = 40, 72
    G = torch.eye(dG, device=DEV, dtype=dtype)
    A = torch.eye(dA, device=DEV, dtype=dtype)
    g = -torch.ones(dG, dA, device=DEV, dtype=dtype)
    w = torch.zeros(dG, dA, device=DEV)
    w[3, 5] = 3.0e38
    ws = kfac.kfac_precondition([kfac.PrecondItem(G, A, g, None, w=w, eta=1e38)])
    assert word(ws) & kfac.ERRW_NONFINITE
    assert math.isinf(float(w[3, 5]))
    assert float(w[0, 0]) == float(torch.tensor(1e38, dtype=torch.float32))
