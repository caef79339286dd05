#!/usr/bin/env python
"""Benchmark of the K-FAC curvature step (factors + damped inverse +
preconditioning) for the ResNet-50 layer set at 32 samples per GPU, on
synthetic inputs with ResNet-50's shapes.

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]
                  [--workload resnet50|conv3x3_256|fc4096|conv3x3_512]

Prints ONE JSON line (rank 0).

Default arm (the CUDA library): inputs resident in HBM; the whole step is
captured once in a CUDA graph and replayed K times between CUDA events
(`value`); each phase is also captured and timed on its own (`phases`).
`e2e` times the same step with the inputs copied from pinned host memory and
the preconditioned gradients copied back inside the timed region.
`schedule` gives the amortised ms per step of the stale-factor schedule
(refresh every k steps) for k in {1, 5, 10, 20}, measured by replaying the
refresh and the precondition-only graphs in that pattern.  For the ResNet-50
workload the line also carries sub-records (`subrecords`: FC 4096, the 3x3
conv, the single FC layer in fp32, the 1024-sample accumulation in 32 chunks)
and the BatchNorm diagonal Fisher (`bn_fisher`).

`--impl reference` runs the CPU oracle (the method's plain fp64 statement)
on the host cores: one whole step, every layer's oracle step timed once
(layers of identical shape are timed once and counted with their
multiplicity), so `value` is the measured time of one full oracle step.

Under torchrun every rank runs an independent replica (the step has no
data-path exchange); the time reported is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time
from collections import Counter

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ResNet-50 K-FAC step ms (factors+inverse+precond); TFLOP/s vs GB300 peak"
NB = 128            # block width of the inversion
SCHEDULE_KS = (1, 5, 10, 20)

# DRAM traffic per launch of a kernel kind from one ncu capture of the same
# kernel build (dram__bytes_read.sum + dram__bytes_write.sum), with the
# profile summary it comes from; None where no capture of the current build
# exists.
_TRAFFIC_SRC = "ncu dram__bytes_read.sum + dram__bytes_write.sum per launch (serialised, cold caches), " \
               "profiles/resnet50_kfac_step_launches.md"
NCU_TRAFFIC = {
    "tc_gemm_tf32x3@inverse": (43.67e6, _TRAFFIC_SRC),
    "inv_diag@inverse": (1.66e6, _TRAFFIC_SRC),
    "inv_prep@inverse": (918.9e6, _TRAFFIC_SRC),
    "im2col@factors": (69.8e6, _TRAFFIC_SRC),
    "tc_gemm_bf16@factors": (2004.1e6, _TRAFFIC_SRC),
    "tc_gemm_bf16@precond": ((330.2e6 + 153.8e6) / 2, _TRAFFIC_SRC),
}


# ------------------------------------------------------------------ workloads

def workload(name):
    from second_order_optimisation_gb300 import workloads as W
    if name == "resnet50":
        return W.resnet50_layers(), 32
    if name == "conv3x3_256":
        return [W.conv_3x3_256()], 32
    if name == "fc4096":
        return [W.fc_4096()], 8192
    if name == "conv3x3_512":   # ResNet-50's last 3x3 conv (A 4608 x 4608, G 512 x 512), 7 x 7, batch 32
        return [L for L in W.resnet50_layers() if L.name == "s4b3_3x3"], 32
    raise SystemExit(f"unknown workload {name}")


def flops(layers, batch):
    """Algorithmic FLOPs of one step: SYRK M d (d + 1) per factor, the
    Cholesky-based inversion d^3 per factor (factor d^3/3, triangular inverse
    d^3/3, product of the inverse factors d^3/3), and the two preconditioning
    products 2 dG^2 dA + 2 dG dA^2 per layer."""
    syrk = inv = pc = 0
    for L in layers:
        M = L.rows(batch)
        syrk += M * L.d_a * (L.d_a + 1) + M * L.d_g * (L.d_g + 1)
        inv += L.d_a ** 3 + L.d_g ** 3
        pc += 2 * L.d_g ** 2 * L.d_a + 2 * L.d_g * L.d_a ** 2
    return dict(syrk=syrk, inv=inv, precond=pc, total=syrk + inv + pc)


def diag_flops(d):
    """FLOPs of the 128 x 128 diagonal blocks of one d x d factor, each
    factored and inverted on CUDA cores (Cholesky + triangular inverse,
    2/3 * 128^3 each block)."""
    return math.ceil(d / NB) * 2 * NB ** 3 // 3


def inversion_split(layers):
    """(tensor-core engine FLOPs, diag-kernel FLOPs) of the inversion."""
    dims = [L.d_a for L in layers] + [L.d_g for L in layers]
    dg = sum(diag_flops(d) for d in dims)
    return sum(d ** 3 for d in dims) - dg, dg


def kernel_work(layers, batch, fl, pk, sm_mhz):
    """Algorithmic work of one step per (phase, kernel kind):
      tc_gemm_bf16 (factors)   SYRK M d(d+1) per factor                   tensor, bf16 peak
      tc_gemm_bf16 (precond)   2 dG^2 dA + 2 dG dA^2 per layer            tensor, bf16 peak
      tc_gemm_tf32x3 (inverse) d^3 - diag blocks' share per factor        tensor, 3 tf32 products
      inv_diag (inverse)       2/3 * 128^3 per 128 x 128 diagonal block   fp32 CUDA cores (alu)
      inv_prep (inverse)       upper triangle of F read (4 B) + the (hi, lo) working pair
                               written below the diagonal 128-blocks and  HBM
                               the diagonal blocks (8 B)
      im2col (factors)         materialised patch bytes written + input read   HBM"""
    tf32x3_peak = pk["bf16"] * (1.1 / 2.25) / 3.0
    # fp32 FMA rate: 152 SMs x 128 lanes x 2 FLOP per cycle at the SM clock
    alu_peak = 152 * 128 * 2 * (sm_mhz or 2070.0) * 1e6 / 1e12
    eng, dgf = inversion_split(layers)
    im2col_bytes = 0
    for L in layers:
        if (L.k > 1 or L.stride > 1) and L.cin % 64 != 0:
            im2col_bytes += L.rows(batch) * L.k * L.k * L.cin * 2 + batch * L.hin * L.hin * L.cin * 2
    pad = lambda d: (d + NB - 1) // NB * NB
    dims = [L.d_a for L in layers] + [L.d_g for L in layers]
    prep_bytes = sum(d * (d + 1) // 2 * 4 + (pad(d) // NB) * (pad(d) // NB - 1) // 2 * NB * NB * 8
                     + pad(d) * NB * 8 for d in dims)
    return {("factors", "tc_gemm_bf16"): (fl["syrk"], "tensor", pk["bf16"], "TFLOP/s", "bf16 burst (measured)"),
            ("precond", "tc_gemm_bf16"): (fl["precond"], "tensor", pk["bf16"], "TFLOP/s", "bf16 burst (measured)"),
            ("inverse", "tc_gemm_tf32x3"): (eng, "tensor", tf32x3_peak, "TFLOP/s",
                                            "measured bf16 burst x 1.1/2.25 (tf32/bf16 nominal) / 3 products"),
            ("inverse", "inv_diag"): (dgf, "alu", alu_peak, "TFLOP/s",
                                      "152 SMs x 128 fp32 lanes x 2 FLOP x SM clock"),
            ("inverse", "inv_prep"): (prep_bytes, "hbm", pk["hbm"], "GB/s", "HBM copy (measured)"),
            ("factors", "im2col"): (im2col_bytes, "hbm", pk["hbm"], "GB/s", "HBM copy (measured)")}


def kernel_rooflines(kern, work, steps, traffic=None):
    """Per-kernel achieved rate from the library's per-launch event timings
    (eager run, each launch bracketed by events on its own stream); DRAM
    traffic per launch from `traffic` (the ResNet-50 step's ncu capture by
    default; other workloads have none)."""
    traffic = NCU_TRAFFIC if traffic is None else traffic
    out = {}
    for ph, ks in kern.items():
        for name, (t, n) in ks.items():
            ms_step = t / steps
            rec = {"ms_per_step": ms_step, "launches_per_step": n / steps, "avg_launch_us": 1e3 * t / max(n, 1)}
            if (ph, name) in work:
                w, bound, peak, unit, psrc = work[(ph, name)]
                scale = 1e12 if unit == "TFLOP/s" else 1e9
                ach = w / (ms_step * 1e-3) / scale if ms_step > 0 else 0.0
                tr = traffic.get(f"{name}@{ph}")
                rec.update({"bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
                            "peak_source": psrc, "work_per_step": w,
                            "traffic": tr[0] if tr else None,
                            "traffic_source": tr[1] if tr else "no ncu capture of this build and workload"})
            out[f"{name}@{ph}"] = rec
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
    """The oracle's whole step for one layer (patches, both factors from I
    with xi = 0.95, pi-split damping, Cholesky-based inverses,
    preconditioning); returns seconds."""
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
    return time.perf_counter() - t0


def shape_key(L):
    return (L.k, L.cin, L.cout, L.stride, L.pad, L.hin, L.hout, L.bias)


def oracle_full_step(layers, batch, tag="bench"):
    """One whole oracle step: each distinct layer shape's step timed once and
    counted with its multiplicity (the oracle's time depends only on the
    shapes).  Returns (seconds, distinct shapes, layers)."""
    counts = Counter(shape_key(L) for L in layers)
    first = {}
    for L in layers:
        first.setdefault(shape_key(L), L)
    total = 0.0
    for key, L in first.items():
        total += counts[key] * oracle_layer_step(L, batch, tag)
    return total, len(first), len(layers)


def cpu_baseline(layers, batch):
    """The oracle as it stands on the host cores: the whole step on all
    cores (measured, distinct shapes once), and the single-thread time of one
    mid-size layer beside its all-core time, which scales the whole step to
    one thread (an estimate, labelled as such)."""
    import oracle
    oracle.build()
    cores = oracle.set_threads(0)
    t_all, nshapes, nlayers = oracle_full_step(layers, batch, "cpu")
    probe = [L for L in layers if L.name == "s3b2_1x1a"] or layers[:1]
    a = oracle_layer_step(probe[0], batch, "cpu1")
    oracle.set_threads(1)
    s = oracle_layer_step(probe[0], batch, "cpu1")
    oracle.set_threads(0)
    return {"value": t_all * 1e3, "unit": "ms", "cores": cores, "kind": "oracle",
            "sample": f"the whole {nlayers}-layer step: every distinct layer shape's oracle step timed once "
                      f"({nshapes} shapes) and counted with its multiplicity; all {cores} host threads",
            "single_thread_ms_estimate": t_all * 1e3 * s / a,
            "single_thread_sample": f"{probe[0].name}: {s * 1e3:.0f} ms on 1 thread vs {a * 1e3:.0f} ms on "
                                    f"{cores}; the whole step scaled by that ratio"}


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


# ------------------------------------------------------------------ reference arm

def run_reference(args, world, rank):
    """One whole oracle step (see oracle_full_step) on rank 0; the other
    ranks exit without work."""
    if rank != 0:
        return 0
    layers, batch = workload(args.workload)
    import oracle
    oracle.build()
    cores = oracle.set_threads(0)
    small = min(layers, key=lambda L: L.d_a ** 3 + L.rows(batch) * L.d_a ** 2)
    for i in range(args.warmup):
        oracle_layer_step(small, batch, tag=f"refw{i}")
    t, nshapes, nlayers = oracle_full_step(layers, batch, "ref")
    ms = t * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": args.gpus,
            "steps": 1, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.workload}_kfac_step", "layers": nlayers, "batch_per_gpu": batch},
            "cpu_baseline": {"value": ms, "unit": "ms", "cores": cores, "kind": "oracle",
                             "sample": f"one whole step ({nlayers} layers; each of the {nshapes} distinct "
                                       f"layer shapes' oracle step timed once and counted with its "
                                       f"multiplicity); --steps {args.steps} requested, one full step timed"},
            "e2e": {"value": ms, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

class Inputs:
    """All inputs of a step packed in ONE pinned host buffer and ONE device
    buffer (256-byte aligned slots), so the end-to-end copy is a single H2D."""

    def __init__(self, layers, batch, dev, tag="bench"):
        import torch

        from second_order_optimisation_gb300 import workloads as W
        host_t, self.slots, off = [], [], 0
        for L in layers:
            x, g, grad = W.layer_inputs(L, batch, tag)
            if L.hin == 1:
                x = x.reshape(x.shape[0], -1)
            ld = (L.d_a + 63) // 64 * 64   # rows on 128-byte boundaries
            gp = torch.zeros(L.d_g, ld, dtype=torch.bfloat16)
            gp[:, :L.d_a] = grad
            for t in (x, g, gp):
                t = t.contiguous()
                host_t.append(t)
                self.slots.append((off, t.shape))
                off += (t.numel() * 2 + 255) // 256 * 256
        self.nbytes = off
        self.layers = layers
        self.hbuf = torch.empty(off, dtype=torch.uint8).pin_memory()
        for t, (o, shp) in zip(host_t, self.slots):
            self.hbuf[o:o + t.numel() * 2].view(torch.bfloat16).view(shp).copy_(t)
        self.dbuf = torch.empty(off, dtype=torch.uint8, device=dev)
        self.dbuf.copy_(self.hbuf, non_blocking=True)
        self.views = self.device_views(self.dbuf)

    def device_views(self, db):
        import torch
        vv = [db[o:o + int(math.prod(shp)) * 2].view(torch.bfloat16).view(shp) for (o, shp) in self.slots]
        return vv[0::3], vv[1::3], [t[:, :L.d_a] for t, L in zip(vv[2::3], self.layers)]


def graph_of(fn, stream):
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_replays(graphs, reps, warmup, stream):
    """ms per repetition of replaying `graphs` in order (CUDA events on the
    launching stream, synchronised on both sides)."""
    import torch
    for _ in range(warmup):
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        for g in graphs:
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def measure(name, steps, warmup, dev, pk, kernels=True):
    """Graph-timed step and phases of one workload, plus the library's
    per-launch event timings (eager).  Returns a dict and the live objects."""
    import torch

    from second_order_optimisation_gb300 import kfac
    from second_order_optimisation_gb300.step import KfacStep
    layers, batch = workload(name)
    inp = Inputs(layers, batch, dev)
    dx, dg, dgr = inp.views
    step = KfacStep(layers, batch, device=dev)
    torch.cuda.synchronize()
    for _ in range(max(warmup, 1)):
        step.run(dx, dg, dgr)
    torch.cuda.synchronize()
    n0 = kfac.launch_count()
    step.run(dx, dg, dgr)
    torch.cuda.synchronize()
    launches = kfac.launch_count() - n0
    assert int(step.info.abs().sum().item()) == 0, "an inversion reported a failing pivot"
    stream = torch.cuda.current_stream()
    kern = {"factors": {}, "inverse": {}, "precond": {}}
    if kernels:
        def add(ph):
            for kname, (t, n) in kfac.timing_read().items():
                a = kern[ph].setdefault(kname, [0.0, 0])
                a[0] += t
                a[1] += n
        kfac.timing_enable(True)
        kfac.timing_read()
        for _ in range(steps):
            step.factor_update(dx, dg)
            add("factors")
            step.damp_invert()
            add("inverse")
            step.precondition(dgr)
            add("precond")
        kfac.timing_enable(False)
        torch.cuda.synchronize()
    g_step = graph_of(lambda: step.run(dx, dg, dgr), stream)
    g_fac = graph_of(lambda: step.factor_update(dx, dg), stream)
    g_inv = graph_of(lambda: step.damp_invert(), stream)
    g_pc = graph_of(lambda: step.precondition(dgr), stream)
    phases = {"factors": time_replays([g_fac], steps, warmup, stream),
              "inverse": time_replays([g_inv], steps, warmup, stream),
              "precond": time_replays([g_pc], steps, warmup, stream)}
    return dict(layers=layers, batch=batch, inp=inp, step=step, stream=stream, launches=launches, kern=kern,
                graphs=dict(step=g_step, precond=g_pc), phases=phases)


def schedule_amortised(m, steps, warmup):
    """Amortised ms per step of the stale-factor schedule: a refresh step
    (the whole step graph) followed by k - 1 precondition-only steps,
    replayed in that pattern."""
    out = {}
    for k in SCHEDULE_KS:
        cycles = max(1, -(-steps // k))
        pattern = [m["graphs"]["step"]] + [m["graphs"]["precond"]] * (k - 1)
        out[f"k{k}"] = time_replays(pattern, cycles, max(1, warmup // k), m["stream"]) / k
    return out


def e2e_time(m, steps, world, dev):
    """Same step with the inputs copied from pinned host memory (one H2D of
    the packed buffer) and all preconditioned gradients copied back (one D2H)
    inside the timed region: torch copies on two copy streams around the
    library calls (the C ABI itself takes device pointers), double-buffered
    so step k's copies overlap the compute of its neighbours.  The library
    calls of each buffer set are captured once in a CUDA graph (as a caller
    that repeats the step would) and replayed."""
    import torch
    step, inp, stream, layers = m["step"], m["inp"], m["stream"], m["layers"]
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
    keep = [s_.out for s_ in step.state]
    dbufs = [inp.dbuf, torch.empty_like(inp.dbuf)]
    in_views = [inp.device_views(db) for db in dbufs]
    graphs = []
    for b in range(2):
        for s_, v in zip(step.state, out_views[b]):
            s_.out = v
        xs_, gs_, grs_ = in_views[b]
        graphs.append(graph_of(lambda: step.run(xs_, gs_, grs_), stream))
    copy, copy_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    f0.record(stream)
    copy.wait_stream(stream)
    with torch.cuda.stream(copy):
        dbufs[0].copy_(inp.hbuf, non_blocking=True)
        ev_in[0].record(copy)
    for k in range(steps):
        b = k % 2
        if k + 1 < steps:
            with torch.cuda.stream(copy):
                if k >= 1:
                    copy.wait_event(ev_done[1 - b])     # step k-1 no longer reads that buffer
                dbufs[1 - b].copy_(inp.hbuf, non_blocking=True)
                ev_in[1 - b].record(copy)
        stream.wait_event(ev_in[b])
        if k >= 2:
            stream.wait_event(ev_out[b])                 # D2H of step k-2 has drained out_dev[b]
        graphs[b].replay()
        ev_done[b].record(stream)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(ev_done[b])
            out_host.copy_(out_dev[b], non_blocking=True)
            ev_out[b].record(copy_out)
    stream.wait_stream(copy)
    stream.wait_stream(copy_out)
    f1.record(stream)
    torch.cuda.synchronize()
    for s_, o in zip(step.state, keep):
        s_.out = o
    return f0.elapsed_time(f1) / steps, inp.nbytes, out_dev[0].numel() * 4


def subrecord(name, steps, warmup, dev, pk, sm_mhz):
    """Graph-timed step and phases of another workload, with the SYRK and
    preconditioner rooflines (as sub-records of the main line)."""
    m = measure(name, steps, warmup, dev, pk)
    ms = time_replays([m["graphs"]["step"]], steps, warmup, m["stream"])
    fl = flops(m["layers"], m["batch"])
    ks = kernel_rooflines(m["kern"], kernel_work(m["layers"], m["batch"], fl, pk, sm_mhz), steps, traffic={})
    keep = ("tc_gemm_bf16@factors", "tc_gemm_bf16@precond", "tc_gemm_tf32x3@inverse", "inv_diag@inverse")
    return {"workload": f"{name}_kfac_step", "ms": ms, "tflops": fl["total"] / (ms * 1e-3) / 1e12,
            "phases_ms": m["phases"], "gpu_launches_per_step": m["launches"],
            "kernels": {k: ks[k] for k in keep if k in ks}}


def fc_small_fp32_record(steps, warmup, dev):
    """The single FC layer in fp32 (a [32, 64] + bias column, g [32, 32];
    factors from I, xi = 0.95, pi-split gamma = 1e-3): the whole step through
    the C ABI, graph-timed, in microseconds (a latency-bound case)."""
    import numpy as np
    import torch

    from second_order_optimisation_gb300 import kfac
    from second_order_optimisation_gb300 import workloads as W
    a, g = W.fc_small_fp32()
    grad = np.concatenate([a, np.ones((32, 1), np.float32)], 1).T @ g / 32.0   # [65, 32] -> G x A below
    ad, gd = torch.from_numpy(a).to(dev), torch.from_numpy(g).to(dev)
    gr = torch.from_numpy(np.ascontiguousarray(grad.T)).to(dev)
    A, G = torch.eye(65, device=dev), torch.eye(32, device=dev)
    Ai, Gi = torch.empty_like(A), torch.empty_like(G)
    out = torch.empty(32, 65, device=dev)
    srcs = [kfac.FactorSource(ad, A, append_one=True, alpha=0.05 / 32, beta=0.95),
            kfac.FactorSource(gd, G, alpha=0.05 / 32, beta=0.95)]
    pairs = [kfac.InvertPair(A, G, Ai, Gi)]
    items = [kfac.PrecondItem(Gi, Ai, gr, out)]
    wf = torch.empty(kfac.kfac_factor_update_workspace_size(srcs), dtype=torch.uint8, device=dev)
    wi = torch.empty(kfac.kfac_damp_invert_workspace_size(pairs), dtype=torch.uint8, device=dev)
    wp = torch.empty(kfac.kfac_precondition_workspace_size(items), dtype=torch.uint8, device=dev)

    def one():
        kfac.kfac_factor_update(srcs, wf)
        kfac.kfac_damp_invert(pairs, 1e-3, workspace=wi)
        kfac.kfac_precondition(items, wp)
    stream = torch.cuda.current_stream()
    g_ = graph_of(one, stream)
    ms = time_replays([g_], max(steps, 20), warmup, stream)
    return {"workload": "fc64x32_fp32_kfac_step", "us": ms * 1e3, "dtype": "f32"}


def accumulation_record(steps, warmup, dev, pk, chunks=32):
    """The ResNet-50 set with factors accumulated over a 1024-sample
    mini-batch in 32 chunks of 32 (beta = xi on the first chunk, 1 after;
    the same seeded chunk re-read each time, 1.38 GB, larger than L2), then
    damped, inverted and applied: graph-timed."""
    import torch
    m = measure("resnet50", 1, 1, dev, pk, kernels=False)
    step, (dx, dg, dgr), stream = m["step"], m["inp"].views, m["stream"]
    rows = [L.rows(m["batch"]) * chunks for L in m["layers"]]

    def acc():
        for c in range(chunks):
            step.factor_update(dx, dg, rows_total=rows, first=(c == 0))
        step.damp_invert()
        step.precondition(dgr)
    g_ = graph_of(acc, stream)
    ms = time_replays([g_], max(1, min(steps, 5)), 1, stream)
    syrk = flops(m["layers"], m["batch"])["syrk"] * chunks
    return {"workload": "resnet50_accum1024_kfac_step", "ms": ms, "chunks": chunks,
            "syrk_tflops": syrk / (ms * 1e-3) / 1e12}


def run_ours(args, world, rank, local):
    import torch

    import __graft_entry__

    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    m = measure(args.workload, args.steps, args.warmup, dev, pk)
    layers, batch, stream = m["layers"], m["batch"], m["stream"]
    fl = flops(layers, batch)
    if args.profile:
        torch.cuda.nvtx.range_push("kfac_step")
        for _ in range(args.steps):
            if args.phase == "inverse":
                m["step"].damp_invert()
            else:
                m["step"].run(*m["inp"].views)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        print(json.dumps({"profile": args.workload, "steps": args.steps,
                          "info_ok": int(m["step"].info.abs().sum().item()) == 0}), flush=True)
        return 0

    # the timed region: K replays of the whole-step graph, clocks sampled meanwhile
    g = m["graphs"]["step"]
    for _ in range(args.warmup):
        g.replay()
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
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    e2e_ms, h2d, d2h = e2e_time(m, args.steps, world, dev)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    sched = schedule_amortised(m, max(args.steps, max(SCHEDULE_KS)), args.warmup)

    kernels = kernel_rooflines(m["kern"], kernel_work(layers, batch, fl, pk, clk.get("sm_mhz")), args.steps)
    dom = max((k for k in kernels if "frac" in kernels[k]), key=lambda k: kernels[k]["ms_per_step"])
    roof = dict(kernels[dom])
    roof["kernel"] = dom
    phases = {n: {"ms": v, "share": v / sum(m["phases"].values())} for n, v in m["phases"].items()}

    subs = None
    bn_line = None
    if args.workload == "resnet50" and not args.no_subrecords:
        subs = {n: subrecord(n, min(args.steps, 10), min(args.warmup, 3), dev, pk, clk.get("sm_mhz"))
                for n in ("fc4096", "conv3x3_256")}
        subs["fc64x32_fp32"] = fc_small_fp32_record(args.steps, args.warmup, dev)
        subs["accum1024"] = accumulation_record(args.steps, args.warmup, dev, pk)
        bn_line = bn_bench(args, dev, stream, pk)

    line = {"metric": METRIC, "value": ms, "unit": "ms", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; ResNet-50 shapes, no ImageNet)",
            "config": {"workload": f"{args.workload}_kfac_step", "layers": len(layers), "batch_per_gpu": batch,
                       "l2": f"inputs larger than L2 ({m['inp'].nbytes / 1e6:.0f} MB per step), no flush",
                       "graph": True, "xi": 0.95, "gamma": 1e-3, "inversion": "fp32 (3 tf32 products)"},
            "tflops": fl["total"] / (ms * 1e-3) / 1e12, "gflop_per_step": fl["total"] / 1e9,
            "phases": phases, "schedule_amortised_ms": sched, "roofline": roof, "kernels": kernels,
            "clocks": clk, "gpu_launches": m["launches"] * args.steps, "gpu_launches_per_step": m["launches"],
            "bn_fisher": bn_line, "subrecords": subs,
            "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": "the library's calls on device buffers (captured once per buffer set in a CUDA "
                           "graph), with torch copies of pinned host buffers inside the timed region: per step "
                           "one H2D of the packed inputs and one D2H of all preconditioned gradients, "
                           "double-buffered on two copy streams"},
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
    ms = time_replays([graph], args.steps, args.warmup, stream)
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
    ap.add_argument("--workload", default="resnet50", choices=("resnet50", "conv3x3_256", "fc4096", "conv3x3_512"))
    ap.add_argument("--phase", default="step", choices=("step", "inverse"),
                    help="with --profile: the NVTX range holds whole steps, or only the damped inversion")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-subrecords", action="store_true")
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
