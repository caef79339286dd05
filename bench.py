#!/usr/bin/env python
"""Benchmark of the K-FAC curvature step (factors + damped inverse +
preconditioning) for the ResNet-50 layer set at 32 samples per GPU, on
synthetic inputs with ResNet-50's shapes.

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]
                  [--workload resnet50|conv3x3_256|fc4096|fc64x32]

Prints ONE JSON line (rank 0).  The default arm times the CUDA library
(device-resident inputs; whole step captured once in a CUDA graph and
replayed); `e2e` times the same step through the C ABI with host buffers
(pinned H2D of the step's inputs and D2H of the preconditioned gradients
inside the timed region).  `--impl reference` times the CPU oracle (the
method's plain fp64 statement) on a bounded sample of the same workload and
scales it to one step by algorithmic FLOPs.  Under torchrun every rank runs
an independent replica (the step has no data-path exchange on one GPU per
replica); the time reported is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ResNet-50 K-FAC step ms (factors+inverse+precond); TFLOP/s vs GB300 peak"
FP32_ALU_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12   # SMs x fp32 lanes x FMA x max clock


# ------------------------------------------------------------------ workloads

def workload(name):
    from second_order_optimisation_gb300 import workloads as W
    if name == "resnet50":
        return W.resnet50_layers(), 32
    if name == "conv3x3_256":
        return [W.conv_3x3_256()], 32
    if name == "fc4096":
        return [W.fc_4096()], 8192
    raise SystemExit(f"unknown workload {name}")


def flops(layers, batch):
    syrk = inv = pc = 0
    for L in layers:
        M = L.rows(batch)
        syrk += M * L.d_a * (L.d_a + 1) + M * L.d_g * (L.d_g + 1)
        inv += L.d_a ** 3 + L.d_g ** 3
        pc += 2 * L.d_g ** 2 * L.d_a + 2 * L.d_g * L.d_a ** 2
    return dict(syrk=syrk, inv=inv, precond=pc, total=syrk + inv + pc)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ------------------------------------------------------------------ clocks

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = [r.split(", ") for r in open(self.f.name).read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip() == "Active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ oracle

def oracle_layer_step(L, batch, tag="bench"):
    """The oracle's full step for one layer (factors from I, EMA, pi damping,
    Cholesky inverses, preconditioning); returns seconds and FLOPs."""
    import numpy as np

    import oracle
    from second_order_optimisation_gb300 import workloads as W
    x, g, grad = W.layer_inputs(L, batch, tag)
    xo = x.float().numpy().astype(np.float64)
    if L.hin == 1:
        xo = xo.reshape(xo.shape[0], -1)
    go = g.float().numpy().astype(np.float64)
    gr = grad.float().numpy().astype(np.float64)
    t0 = time.perf_counter()
    P = oracle.im2col(xo, L.k, L.k, (L.stride,) * 2, (L.pad,) * 2, append_one=L.bias)
    oracle.kfac_layer_step(np.eye(L.d_a), np.eye(L.d_g), P, go, gr, xi=0.95, gamma=1e-3)
    dt = time.perf_counter() - t0
    return dt, flops([L], batch)["total"]


SAMPLE_LAYERS = ("s2b2_3x3", "s3b2_1x1a", "s3b3_3x3")


def cpu_baseline(layers, batch, budget_s=20.0):
    """Oracle on a bounded sample: whole layer steps of a few ResNet-50 layers
    until ~budget_s of CPU work, scaled to one full step by algorithmic FLOPs."""
    import oracle
    cores = oracle.set_threads(0)
    names = [L.name for L in layers]
    sample = [L for L in layers if L.name in SAMPLE_LAYERS] or layers[:1]
    t = f = 0.0
    used = []
    t_start = time.perf_counter()
    for L in sample:
        dt, fl = oracle_layer_step(L, batch)
        t += dt
        f += fl
        used.append(L.name)
        if time.perf_counter() - t_start > budget_s:
            break
    total = flops(layers, batch)["total"]
    ms = t / f * total * 1e3
    return {"value": ms, "unit": "ms", "cores": cores, "kind": "oracle",
            "sample": f"oracle layer steps of {'+'.join(used)} ({f / 1e9:.1f} GFLOP, {t:.1f} s) scaled by "
                      f"algorithmic FLOPs to the {len(names)}-layer step ({total / 1e9:.0f} GFLOP)"}


# ------------------------------------------------------------------ dist

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ arms

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    layers, batch = workload(args.workload)
    import oracle
    oracle.build()
    cores = oracle.set_threads(0)
    sample = [L for L in layers if L.name in SAMPLE_LAYERS] or layers[:1]
    total = flops(layers, batch)["total"]
    ests = []
    for i in range(args.warmup + args.steps):
        L = sample[i % len(sample)]
        dt, fl = oracle_layer_step(L, batch, tag=f"ref{i}")
        if i >= args.warmup:
            ests.append(dt / fl * total * 1e3)
    ms = statistics.mean(ests)
    line = {"impl": "reference", "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.workload}_kfac_step", "layers": len(layers), "batch_per_gpu": batch},
            "cpu_baseline": {"value": ms, "unit": "ms", "cores": cores, "kind": "oracle",
                             "sample": "each step: one oracle layer step cycling over "
                                       f"{'+'.join(L.name for L in sample)}, scaled by algorithmic FLOPs "
                                       f"to the full step ({total / 1e9:.0f} GFLOP)"},
            "e2e": {"value": ms, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import torch

    import __graft_entry__
    from second_order_optimisation_gb300 import kfac
    from second_order_optimisation_gb300 import workloads as W
    from second_order_optimisation_gb300.step import KfacStep

    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    layers, batch = workload(args.workload)
    fl = flops(layers, batch)
    pk = peaks()

    # seeded synthetic inputs, pinned on the host and resident on the device
    hx, hg, hgr, dx, dg, dgr = [], [], [], [], [], []
    for L in layers:
        x, g, grad = W.layer_inputs(L, batch, "bench")
        if L.hin == 1:
            x = x.reshape(x.shape[0], -1)
        ld = (L.d_a + 7) // 8 * 8
        gp = torch.zeros(L.d_g, ld, dtype=torch.bfloat16)
        gp[:, :L.d_a] = grad
        for h, d, t in ((hx, dx, x), (hg, dg, g), (hgr, dgr, gp)):
            h.append(t.contiguous().pin_memory())
            d.append(h[-1].to(dev, non_blocking=True))
    dgr_v = [t[:, :L.d_a] for t, L in zip(dgr, layers)]
    in_bytes = sum(t.numel() * t.element_size() for t in hx + hg + hgr)
    step = KfacStep(layers, batch, device=dev)
    torch.cuda.synchronize()

    # eager warm-up (also sizes and caches the workspaces)
    for _ in range(max(args.warmup, 1)):
        step.run(dx, dg, dgr_v)
    torch.cuda.synchronize()
    if args.profile:
        torch.cuda.nvtx.range_push("kfac_step")
        for _ in range(args.steps):
            step.run(dx, dg, dgr_v)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        print(json.dumps({"profile": args.workload, "steps": args.steps,
                          "info_ok": int(step.info.abs().sum().item()) == 0}), flush=True)
        return 0
    n0 = kfac.launch_count()
    step.run(dx, dg, dgr_v)
    torch.cuda.synchronize()
    launches_per_step = kfac.launch_count() - n0
    assert int(step.info.abs().sum().item()) == 0, "an inversion reported a non-positive pivot"

    # per-phase device times (eager), on the launching stream
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for k in range(args.steps):
        ev[k][0].record(stream)
        step.factor_update(dx, dg)
        ev[k][1].record(stream)
        step.damp_invert()
        ev[k][2].record(stream)
        step.precondition(dgr_v)
        ev[k][3].record(stream)
    torch.cuda.synchronize()
    ph = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in ev)
          for i, n in enumerate(("factors", "inverse", "precond"))}
    eager_ms = statistics.mean(e[0].elapsed_time(e[3]) for e in ev)

    # CUDA graph of one whole step, replayed K times (the timed region)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step.run(dx, dg, dgr_v)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        step.run(dx, dg, dgr_v)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    # end to end through the C ABI with host buffers
    hout = [torch.empty(s.out.shape, dtype=torch.float32).pin_memory() for s in step.state]
    out_bytes = sum(t.numel() * 4 for t in hout)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    f0.record(stream)
    for _ in range(args.steps):
        for h, d in zip(hx + hg + hgr, dx + dg + dgr):
            d.copy_(h, non_blocking=True)
        step.run(dx, dg, dgr_v)
        for h, s in zip(hout, step.state):
            h.copy_(s.out, non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / args.steps, world, dev)

    # roofline of the dominant phase (one kernel type each on the tensor-core path)
    phase_share = {k: v / sum(ph.values()) for k, v in ph.items()}
    dom = max(ph, key=ph.get)
    if dom == "inverse":
        ach = fl["inv"] / (ph["inverse"] * 1e-3) / 1e12
        roof = {"bound": "alu", "kernel": "inversion (sgemm_kernel + leaf_kernel)", "achieved": ach,
                "peak": FP32_ALU_PEAK_TFLOPS, "unit": "TFLOP/s", "frac": ach / FP32_ALU_PEAK_TFLOPS,
                "traffic": None, "peak_src": "derived: 152 SMs x 128 fp32 lanes x 2 x 2.07 GHz"}
    else:
        key = "syrk" if dom == "factors" else "precond"
        ach = fl[key] / (ph[dom] * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "tc_gemm_kernel (" + dom + ")", "achieved": ach,
                "peak": pk["bf16"], "unit": "TFLOP/s", "frac": ach / pk["bf16"], "traffic": None,
                "peak_src": f"{pk['src']} bf16 burst"}
    phases = {}
    for n, key, bound, peak in (("factors", "syrk", "tensor", pk["bf16"]),
                                ("inverse", "inv", "alu", FP32_ALU_PEAK_TFLOPS),
                                ("precond", "precond", "tensor", pk["bf16"])):
        a = fl[key] / (ph[n] * 1e-3) / 1e12
        phases[n] = {"ms": ph[n], "share": phase_share[n], "tflops": a, "bound": bound, "frac": a / peak}

    line = {"metric": METRIC, "value": ms, "unit": "ms", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; ResNet-50 shapes, no ImageNet)",
            "config": {"workload": f"{args.workload}_kfac_step", "layers": len(layers), "batch_per_gpu": batch,
                       "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB per step), no flush",
                       "graph": True, "xi": 0.95, "gamma": 1e-3},
            "tflops": fl["total"] / (ms * 1e-3) / 1e12, "gflop_per_step": fl["total"] / 1e9,
            "eager_ms": eager_ms, "phases": phases, "roofline": roof,
            "clocks": clk, "gpu_launches": launches_per_step * args.steps,
            "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": in_bytes,
                    "d2h_bytes_per_step": out_bytes},
            "wall_s_timed": t_wall}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(layers, batch)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="resnet50")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="eager warm-up, then --steps eager steps inside the NVTX range 'kfac_step' "
                         "(for ncu --nvtx-include kfac_step/); prints no bench line")
    args = ap.parse_args()
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
