"""Writes tests/golden/fc64x32_step.json: the oracle's results for the
single-FC-layer step (a[32,64] fp32 + bias column, g[32,32], factors from I,
xi = 0.95, gamma = 1e-3 split by pi).  Calls only the oracle and the seeded
input generators; rerun it only when the oracle's arithmetic changes for a
reason stated in the commit that changes it."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from second_order_optimisation_gb300 import workloads  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "fc64x32_step.json")


def compute():
    a, g = workloads.fc_small_fp32()
    P = oracle.im2col(a.astype(np.float64), append_one=True)
    grad = oracle.weight_grad(P, g.astype(np.float64), 32)
    r = oracle.kfac_layer_step(np.eye(65), np.eye(32), P, g.astype(np.float64), grad,
                               xi=0.95, gamma=1e-3)
    r["grad"] = grad
    return r


def summary(r):
    rng = np.random.default_rng(0)
    out = {"damp_A": r["damp_A"], "damp_G": r["damp_G"]}
    for k in ("A", "G", "Ainv", "Ginv", "precond", "grad"):
        m = r[k]
        idx = [(int(i), int(j)) for i, j in zip(rng.integers(0, m.shape[0], 24),
                                                 rng.integers(0, m.shape[1], 24))]
        out[k] = {"shape": list(m.shape), "fro": float(np.linalg.norm(m)),
                  "trace": float(np.trace(m)) if m.shape[0] == m.shape[1] else None,
                  "entries": [[i, j, float(m[i, j])] for i, j in idx]}
    return out


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump(summary(compute()), f, indent=1)
    print("wrote", OUT)
