"""kfac_precondition_noalloc: the preconditioner for callers that cannot
allocate device memory (graph capture, synchronisation-free step loops, host
frameworks that own all device memory).  It must give the same results as
kfac_precondition with a caller workspace, on consecutive calls that reuse its
fixed scratch.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from second_order_optimisation_gb300 import kfac, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _items(tag, shapes):
    items = []
    for dG, dA in shapes:
        ld_a, ld_g = (dA + 7) // 8 * 8, (dG + 7) // 8 * 8
        Gi = workloads.normal_f32((dG, dG), 1.0, tag, dG, dA, "G")
        Ai = workloads.normal_f32((dA, dA), 1.0, tag, dG, dA, "A")
        gr = workloads.normal_f32((dG, dA), 1e-3, tag, dG, dA, "g")
        Gd = torch.zeros(dG, ld_g, dtype=torch.bfloat16, device=DEV)
        Ad = torch.zeros(dA, ld_a, dtype=torch.bfloat16, device=DEV)
        gd = torch.zeros(dG, ld_a, dtype=torch.bfloat16, device=DEV)
        Gd[:, :dG] = workloads.to_bf16((Gi + Gi.T) / 2).to(DEV)
        Ad[:, :dA] = workloads.to_bf16((Ai + Ai.T) / 2).to(DEV)
        gd[:, :dA] = workloads.to_bf16(gr).to(DEV)
        items.append((Gd[:, :dG], Ad[:, :dA], gd[:, :dA]))
    return items


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    lib = kfac.load()
    assert lib.kfac_noalloc_scratch_bytes() == 32 << 20
    for call, shapes in enumerate(([(256, 576), (64, 147), (300, 700)], [(512, 1152), (130, 300)])):
        items = _items(f"noalloc{call}", shapes)
        # the whole scratch of the call (intermediate, tensor maps, split-K
        # partial tiles) must fit the fixed array
        need = kfac.kfac_precondition_workspace_size(
            [kfac.PrecondItem(G, A, g, torch.empty(g.shape, device=DEV)) for G, A, g in items])
        assert need <= lib.kfac_noalloc_scratch_bytes()
        ref = [torch.empty(it[2].shape, device=DEV) for it in items]
        out = [torch.full(it[2].shape, float("nan"), device=DEV) for it in items]
        kfac.kfac_precondition([kfac.PrecondItem(G, A, g, o) for (G, A, g), o in zip(items, ref)])
        kfac.kfac_precondition_noalloc([kfac.PrecondItem(G, A, g, o) for (G, A, g), o in zip(items, out)])
        torch.cuda.synchronize()
        for o, r in zip(out, ref):
            o, r = o.double().cpu().numpy(), r.double().cpu().numpy()
            assert np.all(np.isfinite(o))
            assert np.linalg.norm(o - r) <= 2e-2 * np.linalg.norm(r)


def test_noalloc_rejects_oversized_calls():
    lib = kfac.load()
    dG, dA = 4096, 4104                       # needs more than 32 MiB of scratch
    G = torch.zeros(dG, dG, dtype=torch.bfloat16, device=DEV)
    A = torch.zeros(dA, dA, dtype=torch.bfloat16, device=DEV)
    g = torch.zeros(dG, dA, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(dG, dA, device=DEV)
    arr = kfac._precond_descs([kfac.PrecondItem(G, A, g, out)])
    assert lib.kfac_precondition_noalloc(arr, 1, kfac.KFAC_BF16, None) == kfac.KFAC_ERR_WORKSPACE
