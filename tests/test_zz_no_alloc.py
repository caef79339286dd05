"""kfac_precondition_noalloc: the preconditioner for callers that cannot
allocate device memory (host frameworks that own all device memory through
their own pool, step loops that cannot take cudaMalloc's implicit device-wide
synchronisation, callers with a device-memory budget fixed at start-up).

It runs the same kernels as kfac_precondition, only with the library's fixed
device scratch in place of the caller's workspace, so its outputs must be
bitwise the same -- on two calls in a row, which reuse the scratch and its
left-over contents.  This file is collected last on purpose: if it fails, a
run that stops at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from second_order_optimisation_gb300 import kfac, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _items(tag, shapes, dtype):
    """(G_inv, A_inv, grad) per layer: symmetric seeded inverses and a
    1e-3-scale gradient; bf16 operands get leading dimensions rounded up to 8."""
    items = []
    for dG, dA in shapes:
        Gi = workloads.normal_f32((dG, dG), 1.0, tag, dG, dA, "G")
        Ai = workloads.normal_f32((dA, dA), 1.0, tag, dG, dA, "A")
        gr = workloads.normal_f32((dG, dA), 1e-3, tag, dG, dA, "g")
        Gi, Ai = (Gi + Gi.T) / 2, (Ai + Ai.T) / 2
        if dtype == torch.bfloat16:
            ld_a, ld_g = (dA + 7) // 8 * 8, (dG + 7) // 8 * 8
            Gd = torch.zeros(dG, ld_g, dtype=dtype, device=DEV)
            Ad = torch.zeros(dA, ld_a, dtype=dtype, device=DEV)
            gd = torch.zeros(dG, ld_a, dtype=dtype, device=DEV)
            Gd[:, :dG] = workloads.to_bf16(Gi).to(DEV)
            Ad[:, :dA] = workloads.to_bf16(Ai).to(DEV)
            gd[:, :dA] = workloads.to_bf16(gr).to(DEV)
            items.append((Gd[:, :dG], Ad[:, :dA], gd[:, :dA]))
        else:
            items.append(tuple(torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (Gi, Ai, gr)))
    return items


CALLS = {
    torch.bfloat16: ([(256, 576), (64, 147), (300, 700)], [(512, 1152), (130, 300)]),
    torch.float32: ([(64, 147), (200, 300)], [(130, 257), (32, 65)]),
}


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_noalloc_equals_workspace_entry_point_on_two_calls(dtype):
    lib = kfac.load()
    assert lib.kfac_noalloc_scratch_bytes() == 32 << 20
    for call, shapes in enumerate(CALLS[dtype]):
        items = _items(f"noalloc{call}", shapes, dtype)
        # all scratch of the call (intermediate, tensor maps, split-K partial
        # tiles) fits the fixed array
        need = kfac.kfac_precondition_workspace_size(
            [kfac.PrecondItem(G, A, g, torch.empty(g.shape, device=DEV)) for G, A, g in items])
        assert 0 < need <= lib.kfac_noalloc_scratch_bytes()
        ref = [torch.full(it[2].shape, float("nan"), device=DEV) for it in items]
        out = [torch.full(it[2].shape, float("nan"), device=DEV) for it in items]
        kfac.kfac_precondition([kfac.PrecondItem(G, A, g, o) for (G, A, g), o in zip(items, ref)])
        kfac.kfac_precondition_noalloc([kfac.PrecondItem(G, A, g, o) for (G, A, g), o in zip(items, out)])
        torch.cuda.synchronize()
        for (G, A, g), o, r in zip(items, out, ref):
            assert torch.isfinite(r).all()
            assert torch.equal(o, r), float((o - r).abs().max())
            # and both are the preconditioned gradient itself (fp64 product of
            # the operands as stored; bf16 operands round the intermediate)
            exp = G.double().cpu() @ g.double().cpu() @ A.double().cpu()
            tol = 2e-2 if dtype == torch.bfloat16 else 1e-4
            assert float((o.double().cpu() - exp).norm() / exp.norm()) <= tol


def test_noalloc_rejects_oversized_calls():
    lib = kfac.load()
    dG, dA = 4096, 4104                       # needs more than 32 MiB of scratch
    G = torch.zeros(dG, dG, dtype=torch.bfloat16, device=DEV)
    A = torch.zeros(dA, dA, dtype=torch.bfloat16, device=DEV)
    g = torch.zeros(dG, dA, dtype=torch.bfloat16, device=DEV)
    out = torch.full((dG, dA), 7.0, device=DEV)
    arr = kfac._precond_descs([kfac.PrecondItem(G, A, g, out)])
    assert kfac.kfac_precondition_workspace_size([kfac.PrecondItem(G, A, g, out)]) > lib.kfac_noalloc_scratch_bytes()
    assert lib.kfac_precondition_noalloc(arr, 1, kfac.KFAC_BF16, None) == kfac.KFAC_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())           # nothing was enqueued
