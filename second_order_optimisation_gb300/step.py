"""One K-FAC curvature step over a layer set, through the C ABI.

`KfacStep` owns the per-layer state (running factors A, G; damped inverses in
fp32 and bf16; preconditioned gradients) and the three workspaces, all
allocated once on the device.  `run()` enqueues the hot path of Osawa et al.
(section 3.2, Eq. 5-7) for every layer on the current stream:

    kfac_factor_update  (A from the layer inputs, G from the output grads,
                         running average with xi, all layers in one call)
    kfac_damp_invert    (pi-split Tikhonov damping, all layers in one call)
    kfac_precondition   (G^-1 grad A^-1, all layers in one call)

Inputs are the per-layer bf16 tensors x (NHWC), g ([M, C_out]) and grad
([C_out, d_A]); with `rows_total` the statistic of several chunks of a larger
mini-batch can be accumulated before the inversion (gradient accumulation,
section 2).

`step()` runs the same phases under the stale-factor schedule of the paper's
contributions list (section 1: after a few hundred iterations the Fisher is
updated less often).  The pages give no period, so it is a parameter: steps
t < warmup refresh the factors and their inverses every time; after that only
every `update_every`-th step does ((t - warmup) % update_every == 0), and the
other steps precondition with the inverses of the last refresh.  A stale step
skips the factor statistic as well as the inversion (the factors are
"updated" less often, not only inverted less often).  With `weights` the
preconditioner also applies w <- w - eta * P in its epilogue (Eq. 8).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

from . import kfac
from .workloads import Layer


def _pitch(d: int) -> int:
    """Row pitch (elements) of the step's matrices: rows start on 128-byte
    boundaries (16-bit) / 256-byte boundaries (fp32), which the tensor-memory
    copies read in whole 128-byte segments (FC 4096's preconditioner: 0.36 ->
    0.31 ms against rows padded to 8 elements only)."""
    return (d + 63) // 64 * 64


def _matrix(rows: int, cols: int, device, dtype=torch.float32, eye: bool = False) -> torch.Tensor:
    """A [rows, cols] view of a buffer with row pitch _pitch(cols)."""
    v = torch.zeros(rows, _pitch(cols), dtype=dtype, device=device)[:, :cols]
    if eye:
        v.copy_(torch.eye(rows, cols, dtype=dtype, device=device))
    return v


@dataclass
class LayerState:
    layer: Layer
    A: torch.Tensor
    G: torch.Tensor
    A_inv: torch.Tensor
    G_inv: torch.Tensor
    A_inv16: torch.Tensor      # [dA, dA] bf16 view (row pitch _pitch(dA))
    G_inv16: torch.Tensor
    out: torch.Tensor          # preconditioned gradient [dG, dA] fp32


class KfacStep:
    def __init__(self, layers: Sequence[Layer], batch: int, xi: float = 0.95, gamma: float = 1e-3,
                 device="cuda", update_every: int = 1, warmup: int = 0,
                 weights: Optional[Sequence[torch.Tensor]] = None, eta: float = 0.0):
        self.layers = list(layers)
        self.batch = batch
        self.xi = xi
        self.gamma = gamma
        self.device = torch.device(device)
        if update_every < 1 or warmup < 0:
            raise ValueError("update_every must be >= 1 and warmup >= 0")
        self.update_every = int(update_every)
        self.warmup = int(warmup)
        self.t = 0                  # steps taken by step()
        if weights is not None and len(weights) != len(self.layers):
            raise ValueError("one weight tensor per layer")
        self.weights = list(weights) if weights is not None else None
        self.eta = float(eta)
        self.state: List[LayerState] = []
        for L in self.layers:
            dA, dG = L.d_a, L.d_g
            self.state.append(LayerState(
                L,
                _matrix(dA, dA, self.device, eye=True), _matrix(dG, dG, self.device, eye=True),
                _matrix(dA, dA, self.device), _matrix(dG, dG, self.device),
                _matrix(dA, dA, self.device, torch.bfloat16), _matrix(dG, dG, self.device, torch.bfloat16),
                _matrix(dG, dA, self.device)))
        self.info = torch.zeros(2 * len(self.layers), dtype=torch.int32, device=self.device)
        self.damp = torch.zeros(2 * len(self.layers), device=self.device)
        self._ws = {}

    # ---------------------------------------------------------------- pieces
    def reset_factors(self):
        for s in self.state:
            s.A.copy_(torch.eye(s.A.shape[0], device=self.device))
            s.G.copy_(torch.eye(s.G.shape[0], device=self.device))

    def factor_sources(self, xs, gs, rows_total: Optional[Sequence[int]] = None, first: bool = True):
        srcs = []
        for i, (s, x, g) in enumerate(zip(self.state, xs, gs)):
            L = s.layer
            M = rows_total[i] if rows_total is not None else L.rows(self.batch)
            alpha = (1.0 - self.xi) / M
            beta = self.xi if first else 1.0
            if L.name == "fc" or (L.hin == 1 and L.k == 1):
                xa = x.reshape(x.shape[0], -1)
            else:
                xa = x
            srcs.append(kfac.FactorSource(xa, s.A, L.k, L.k, (L.stride, L.stride), (L.pad, L.pad),
                                          L.bias, alpha, beta))
            srcs.append(kfac.FactorSource(g, s.G, alpha=alpha, beta=beta))
        return srcs

    def invert_pairs(self):
        return [kfac.InvertPair(s.A, s.G, s.A_inv, s.G_inv, s.A_inv16, s.G_inv16) for s in self.state]

    def precond_items(self, grads):
        ws = self.weights if self.weights is not None else [None] * len(self.state)
        return [kfac.PrecondItem(s.G_inv16, s.A_inv16, gr, s.out,
                                 w=w, eta=self.eta)
                for s, gr, w in zip(self.state, grads, ws)]

    def _workspace(self, key, nbytes):
        w = self._ws.get(key)
        if w is None or w.numel() < nbytes:
            w = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            self._ws[key] = w
        return w

    # ---------------------------------------------------------------- phases
    def factor_update(self, xs, gs, rows_total=None, first=True, stream=None):
        srcs = self.factor_sources(xs, gs, rows_total, first)
        ws = self._workspace("factor", kfac.kfac_factor_update_workspace_size(srcs))
        kfac.kfac_factor_update(srcs, ws, stream)

    def damp_invert(self, stream=None):
        pairs = self.invert_pairs()
        ws = self._workspace("invert", kfac.kfac_damp_invert_workspace_size(pairs))
        kfac.kfac_damp_invert(pairs, self.gamma, True, self.info, self.damp, ws, stream)

    def precondition(self, grads, stream=None):
        items = self.precond_items(grads)
        ws = self._workspace("precond", kfac.kfac_precondition_workspace_size(items))
        kfac.kfac_precondition(items, ws, stream)

    def run(self, xs, gs, grads, stream=None):
        """One full step: factors + inverse + preconditioning for all layers."""
        self.factor_update(xs, gs, stream=stream)
        self.damp_invert(stream)
        self.precondition(grads, stream)

    # ---------------------------------------------------------------- schedule
    def refresh_due(self, t: Optional[int] = None) -> bool:
        """Whether step t (default: the next one) refreshes factors and inverses."""
        t = self.t if t is None else t
        return t < self.warmup or (t - self.warmup) % self.update_every == 0

    def step(self, xs, gs, grads, stream=None) -> bool:
        """Step t of the stale-factor schedule; returns whether it refreshed.
        xs / gs are only read on refresh steps (None is accepted otherwise)."""
        refresh = self.refresh_due()
        if refresh:
            self.factor_update(xs, gs, stream=stream)
            self.damp_invert(stream)
        self.precondition(grads, stream)
        self.t += 1
        return refresh
