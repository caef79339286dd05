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


def schur_gemm_flops(d, leaf=128, leaf_max=256):
    """Useful fp32 flops of the tensor-core Schur-complement GEMMs that invert
    one d x d factor (padded to a multiple of 128, split on 128-row block
    boundaries down to leaves of 128 or 256 rows; the two symmetric updates
    count half)."""
    def rec(n):
        if n <= leaf or n == leaf_max:
            return 0
        nb = n // leaf
        h = leaf * (nb // 2)
        m = n - h
        return rec(h) + rec(m) + 2 * h * m * h + m * m * h + 2 * h * m * m + h * h * m
    dp = -(-d // leaf) * leaf
    return rec(dp)


def leaf_sizes(d, leaf=128, leaf_max=256):
    """Block sizes of the leaves that invert one d x d factor."""
    out = []
    def rec(n):
        if n <= leaf or n == leaf_max:
            out.append(n)
            return
        nb = n // leaf
        h = leaf * (nb // 2)
        rec(h)
        rec(n - h)
    rec(-(-d // leaf) * leaf)
    return out


def leaf_flops(n):
    """Gauss-Jordan inverse of an n x n block: n^3 multiply-adds (2 n^3 flops)."""
    return 2 * n ** 3


def kernel_rooflines(kern, layers, batch, fl, pk, steps):
    """Per-kernel achieved rate vs its roofline from the per-phase event
    totals.  Algorithmic work per step:
      tc_gemm_bf16 (factors)  SYRK M*d(d+1) per factor            (tensor, bf16 peak)
      tc_gemm_bf16 (precond)  2 dG^2 dA + 2 dG dA^2 per layer      (tensor, bf16 peak)
      tc_gemm_tf32x3          Schur GEMM flops (schur_gemm_flops)  (tensor, tf32 peak / 3 products)
      inv_leaf                2 n^3 per n-block leaf (n = 128, 256)  (tensor, tf32 peak / 3 products)
      im2col                  bytes of the materialised patch matrices written + inputs read (HBM)
      inv_prep                upper triangle of F read (4 B) + the (hi, lo) pair written, dp^2 x 8 B
      inv_finish              upper triangle of the pair read (8 B) + fp32 and bf16 inverses written
                              (d^2 x 6 B)                          (HBM)"""
    tf32x3_peak = pk["bf16"] * (1.1 / 2.25) / 3.0
    schur = sum(schur_gemm_flops(L.d_a) + schur_gemm_flops(L.d_g) for L in layers)
    leaves = sum(leaf_flops(n) for L in layers for d in (L.d_a, L.d_g) for n in leaf_sizes(d))
    im2col_bytes = 0
    for L in layers:
        # patches are materialised only where the SYRK cannot read the input
        # through an im2col tensor map (channels not in whole 64-wide taps)
        if (L.k > 1 or L.stride > 1) and L.cin % 64 != 0:
            im2col_bytes += L.rows(batch) * L.k * L.k * L.cin * 2 + batch * L.hin * L.hin * L.cin * 2
    pad = lambda d: (d + 127) // 128 * 128
    dims = [L.d_a for L in layers] + [L.d_g for L in layers]
    prep_bytes = sum(d * (d + 1) // 2 * 4 + pad(d) ** 2 * 8 for d in dims)
    finish_bytes = sum(d * (d + 1) // 2 * 8 + d * d * 6 for d in dims)
    work = {("factors", "tc_gemm_bf16"): (fl["syrk"], "tensor", pk["bf16"], "TFLOP/s"),
            ("inverse", "inv_prep"): (prep_bytes, "hbm", pk["hbm"], "GB/s"),
            ("inverse", "inv_finish"): (finish_bytes, "hbm", pk["hbm"], "GB/s"),
            ("precond", "tc_gemm_bf16"): (fl["precond"], "tensor", pk["bf16"], "TFLOP/s"),
            ("inverse", "tc_gemm_tf32x3"): (schur, "tensor", tf32x3_peak, "TFLOP/s"),
            ("inverse", "inv_leaf"): (leaves, "tensor", tf32x3_peak, "TFLOP/s"),
            ("factors", "im2col"): (im2col_bytes, "hbm", pk["hbm"], "GB/s")}
    out = {}
    for ph, ks in kern.items():
        for name, (t, n) in ks.items():
            key = f"{name}@{ph}"
            ms_step = t / steps
            rec = {"ms_per_step": ms_step, "launches_per_step": n / steps,
                   "avg_launch_us": 1e3 * t / max(n, 1)}
            if (ph, name) in work:
                w, bound, peak, unit = work[(ph, name)]
                scale = 1e12 if unit == "TFLOP/s" else 1e9
                ach = w / (ms_step * 1e-3) / scale
                rec.update({"bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
                            "traffic": None})
            out[key] = rec
    return out


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
    import numpy as np
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
    # all inputs of a step packed in ONE pinned host buffer and ONE device
    # buffer (256-byte aligned slots), so the end-to-end copy is a single H2D
    host_t, slots, off = [], [], 0
    for L in layers:
        x, g, grad = W.layer_inputs(L, batch, "bench")
        if L.hin == 1:
            x = x.reshape(x.shape[0], -1)
        ld = (L.d_a + 7) // 8 * 8
        gp = torch.zeros(L.d_g, ld, dtype=torch.bfloat16)
        gp[:, :L.d_a] = grad
        for t in (x, g, gp):
            t = t.contiguous()
            host_t.append(t)
            slots.append((off, t.shape))
            off += (t.numel() * 2 + 255) // 256 * 256
    in_bytes = off
    hbuf = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    hv, dv = [], []
    for t, (o, shp) in zip(host_t, slots):
        n = t.numel() * 2
        h = hbuf[o:o + n].view(torch.bfloat16).view(shp)
        h.copy_(t)
        hv.append(h)
        dv.append(dbuf[o:o + n].view(torch.bfloat16).view(shp))
    del host_t
    dbuf.copy_(hbuf, non_blocking=True)
    dx, dg, dgr = dv[0::3], dv[1::3], dv[2::3]
    dgr_v = [t[:, :L.d_a] for t, L in zip(dgr, layers)]
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

    # per-phase device times (eager), on the launching stream, and every
    # library kernel timed with CUDA events by the library's timing hooks
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    kern = {"factors": {}, "inverse": {}, "precond": {}}

    def add(ph):
        for name, (t, n) in kfac.timing_read().items():
            a = kern[ph].setdefault(name, [0.0, 0])
            a[0] += t
            a[1] += n

    kfac.timing_enable(True)
    kfac.timing_read()
    for k in range(args.steps):
        ev[k][0].record(stream)
        step.factor_update(dx, dg)
        ev[k][1].record(stream)
        add("factors")
        step.damp_invert()
        ev[k][2].record(stream)
        add("inverse")
        step.precondition(dgr_v)
        ev[k][3].record(stream)
        add("precond")
    kfac.timing_enable(False)
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

    # end to end through the C ABI with host buffers: every step copies its
    # inputs (one pinned H2D of the packed buffer) and reads back every
    # preconditioned gradient (one D2H); the H2D and the D2H run on two more
    # streams, double buffered, so step k's copies overlap the compute of its
    # neighbours and each other (the host link carries both directions at once)
    out_sizes = [s.out.numel() for s in step.state]
    out_dev = [torch.empty(sum(out_sizes), device=dev) for _ in range(2)]
    out_host = torch.empty(sum(out_sizes)).pin_memory()
    out_views = []
    for od in out_dev:
        vs, o = [], 0
        for s_, n in zip(step.state, out_sizes):
            vs.append(od[o:o + n].view(s_.out.shape))
            o += n
        out_views.append(vs)
    dbufs = [dbuf, torch.empty_like(dbuf)]
    in_views = []
    for db in dbufs:
        vv = [db[o:o + int(np.prod(shp)) * 2].view(torch.bfloat16).view(shp) for (o, shp) in slots]
        in_views.append((vv[0::3], vv[1::3], [t[:, :L.d_a] for t, L in zip(vv[2::3], layers)]))
    out_bytes = out_dev[0].numel() * 4
    copy = torch.cuda.Stream()
    copy_out = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    f0.record(stream)
    copy.wait_stream(stream)
    with torch.cuda.stream(copy):
        dbufs[0].copy_(hbuf, non_blocking=True)
        ev_in[0].record(copy)
    for k in range(args.steps):
        b = k % 2
        if k + 1 < args.steps:
            with torch.cuda.stream(copy):
                if k >= 1:
                    copy.wait_event(ev_done[1 - b])     # step k-1 no longer reads that buffer
                dbufs[1 - b].copy_(hbuf, non_blocking=True)
                ev_in[1 - b].record(copy)
        stream.wait_event(ev_in[b])
        if k >= 2:
            stream.wait_event(ev_out[b])                 # D2H of step k-2 has drained out_dev[b]
        for s_, v in zip(step.state, out_views[b]):
            s_.out = v
        xs_, gs_, grs_ = in_views[b]
        step.run(xs_, gs_, grs_)
        ev_done[b].record(stream)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(ev_done[b])
            out_host.copy_(out_dev[b], non_blocking=True)
            ev_out[b].record(copy_out)
    stream.wait_stream(copy)
    stream.wait_stream(copy_out)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / args.steps, world, dev)

    # BatchNorm diagonal Fisher of the 53 BN layers, per-sample scale and
    # shift gradients [1024, C] fp32 (the large-mini-batch accumulation case)
    bn_line = bn_bench(args, dev, stream, pk) if args.workload == "resnet50" else None

    # per-kernel rooflines from the live event timings; the dominant kernel
    # (largest share of the step's device time) goes in "roofline"
    kernels = kernel_rooflines(kern, layers, batch, fl, pk, args.steps)
    dom_name = max(kernels, key=lambda k: kernels[k]["ms_per_step"])
    roof = dict(kernels[dom_name])
    roof["kernel"] = dom_name
    phase_share = {k: v / sum(ph.values()) for k, v in ph.items()}
    phases = {n: {"ms": ph[n], "share": phase_share[n]} for n in ph}

    line = {"metric": METRIC, "value": ms, "unit": "ms", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; ResNet-50 shapes, no ImageNet)",
            "config": {"workload": f"{args.workload}_kfac_step", "layers": len(layers), "batch_per_gpu": batch,
                       "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB per step), no flush",
                       "graph": True, "xi": 0.95, "gamma": 1e-3},
            "tflops": fl["total"] / (ms * 1e-3) / 1e12, "gflop_per_step": fl["total"] / 1e9,
            "eager_ms": eager_ms, "phases": phases, "roofline": roof, "kernels": kernels,
            "clocks": clk, "gpu_launches": launches_per_step * args.steps, "bn_fisher": bn_line,
            "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": in_bytes,
                    "d2h_bytes_per_step": out_bytes,
                    "how": "C ABI calls with host buffers; per step one pinned H2D of the packed inputs and "
                           "one D2H of all preconditioned gradients, double-buffered on two copy streams (H2D, D2H)"},
            "wall_s_timed": t_wall}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(layers, batch)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def bn_bench(args, dev, stream, pk, nsamples=1024):
    import torch

    from second_order_optimisation_gb300 import kfac
    from second_order_optimisation_gb300 import workloads as W
    chans = W.resnet50_bn_channels()
    items = []
    for xg, xb in W.bn_grads(chans, nsamples, "bench_bn"):
        for x in (xg, xb):
            C = x.shape[1]
            items.append(kfac.BnItem(torch.from_numpy(x).to(dev), torch.empty(C, device=dev),
                                     torch.empty(C, device=dev), torch.empty(C, device=dev)))
    read = sum(it.x.numel() * 4 for it in items)
    written = sum(3 * it.F.numel() * 4 for it in items)
    kfac.kfac_bn_diag_fisher(items, 1e-3)           # warm (and host set-up) outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()                   # one launch per replay, no host overhead inside
    with torch.cuda.graph(graph):
        kfac.kfac_bn_diag_fisher(items, 1e-3)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    gbs = (read + written) / (ms * 1e-3) / 1e9
    return {"layers": len(chans), "tensors": len(items), "n_samples": nsamples, "ms": ms,
            "bytes": read + written, "achieved_gbs": gbs, "peak_gbs": pk["hbm"], "frac": gbs / pk["hbm"],
            "bound": "hbm", "l2": "inputs larger than L2 (%.0f MB), no flush" % (read / 1e6)}


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
