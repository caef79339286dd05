"""The N > 1 path of bench.py on the CPU (gloo, world size 2): ranks are
independent replicas; the reported time is the max over ranks, reduced with
one all-reduce of a float, and only rank 0 prints a line (the reference arm's
other ranks exit without work)."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import argparse
    import contextlib
    import io

    import bench
    args = argparse.Namespace(impl="reference", gpus=world, steps=1, warmup=0, workload="resnet50")
    w, r, local = bench.dist_setup(args)
    try:
        got = bench.max_over_ranks(float(10 * (rank + 1)), w, "cpu")
        bench.barrier(w)
        out = io.StringIO()
        rc = None
        if r != 0:   # rank 0 would time the whole oracle step; the others must return at once
            with contextlib.redirect_stdout(out):
                rc = bench.run_reference(args, w, r)
        q.put((r, w, got, rc, out.getvalue()))
    finally:
        import torch.distributed as dist
        dist.destroy_process_group()


def test_two_replicas_reduce_max_and_only_rank0_prints():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    assert [x[:3] for x in res] == [(0, 2, 20.0), (1, 2, 20.0)]
    assert res[1][3] == 0 and res[1][4] == ""
