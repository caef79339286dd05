"""GPU parity of the stale-factor schedule and the fused step on the weights.

Osawa et al., section 1 (contributions): after a warm-up the Fisher is
updated less often.  KfacStep.step() refreshes the factors and their inverses
on steps t < warmup and on every update_every-th step after, and otherwise
preconditions with the inverses of the last refresh; with weights it also
applies w <- w - eta * P (section 3.2, Eq. 8) in the preconditioner's
epilogue.  Each step's preconditioned gradient is compared with the oracle's
run of the same schedule on the same seeded inputs (relative Frobenius error
<= 2e-2, bf16 inputs), and the weights after the last step with the oracle's
w0 - eta * sum of its preconditioned gradients.
"""
import numpy as np
import pytest
import torch

import oracle
from second_order_optimisation_gb300 import workloads
from second_order_optimisation_gb300.step import KfacStep

pytestmark = pytest.mark.gpu
DEV = "cuda"
XI, GAMMA, ETA = 0.95, 1e-3, 0.05

LAYERS = [workloads.Layer("c3x3_64_96", 64, 96, 3, 1, 1, 10, 10),
          workloads.Layer("fc300_130", 300, 130, 1, 1, 0, 1, 1, bias=True)]


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / (nb if nb > 0 else 1.0))


def grad_dev(w):
    dG, dA = w.shape
    buf = torch.zeros(dG, (dA + 7) // 8 * 8, dtype=w.dtype, device=DEV)
    buf[:, :dA] = w.to(DEV)
    return buf[:, :dA]


def patches(L, x):
    xa = x.float().numpy()
    if L.hin == 1 and L.k == 1:
        return oracle.im2col(xa.reshape(xa.shape[0], -1), append_one=L.bias)
    return oracle.im2col(xa, L.k, L.k, (L.stride, L.stride), (L.pad, L.pad), append_one=L.bias)


@pytest.mark.parametrize("warmup,every,nsteps", [(1, 2, 6), (0, 3, 7), (2, 1, 4)],
                         ids=["warmup1-every2", "warmup0-every3", "every-step"])
def test_stale_schedule_matches_oracle(warmup, every, nsteps):
    batch = 8
    w0 = [workloads.normal_f32((L.d_g, L.d_a), 5e-2, "sched-w", L.name) for L in LAYERS]
    weights = [torch.from_numpy(w).to(DEV) for w in w0]
    step = KfacStep(LAYERS, batch, xi=XI, gamma=GAMMA, update_every=every, warmup=warmup,
                    weights=weights, eta=ETA)
    host = {L.name: [] for L in LAYERS}
    outs = {L.name: [] for L in LAYERS}
    refreshed = []
    last_A = None
    for t in range(nsteps):
        xs, gs, grads = [], [], []
        for L in LAYERS:
            x, g, w = workloads.layer_inputs(L, batch, "sched", warmup, every, t)
            host[L.name].append((patches(L, x), g.float().numpy(), w.float().numpy()))
            xs.append(x.to(DEV))
            gs.append(g.to(DEV))
            grads.append(grad_dev(w))
        due = step.refresh_due()
        assert due == oracle.is_refresh_step(t, warmup, every)
        refreshed.append(step.step(xs, gs, grads))
        torch.cuda.synchronize()
        A_now = step.state[0].A.clone()
        if not refreshed[-1]:
            assert torch.equal(A_now, last_A), "a stale step changed the factors"
        last_A = A_now
        for L, s in zip(LAYERS, step.state):
            outs[L.name].append(f64(s.out))
    assert int(step.info.abs().sum().item()) == 0
    assert refreshed == [bool(oracle.is_refresh_step(t, warmup, every)) for t in range(nsteps)]
    for i, L in enumerate(LAYERS):
        ref = oracle.kfac_schedule(np.eye(L.d_a), np.eye(L.d_g), host[L.name], XI, GAMMA, warmup, every)
        for t in range(nsteps):
            assert rel(outs[L.name][t], ref[t]) <= 2e-2, (L.name, t, rel(outs[L.name][t], ref[t]))
        w_ref = w0[i].astype(np.float64)
        for P in ref:
            w_ref = oracle.weight_update(w_ref, P, ETA)
        got = f64(weights[i])
        assert rel(got - w0[i], w_ref - w0[i]) <= 2e-2, (L.name, rel(got - w0[i], w_ref - w0[i]))
