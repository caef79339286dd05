"""CPU oracle for the K-FAC curvature step (test infrastructure only).

Plain double-precision C (``kfac_oracle.c``) loaded through ctypes.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the CUDA library never does, and the two
share no code.  Every function takes and returns numpy float64 arrays; inputs
stored as bf16 or fp32 are widened exactly before they get here.

Source: Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
Kronecker-Factored Approximate Curvature for Deep Convolutional Neural
Networks", section 3.2 (Eq. 4-7) and section 1 (diagonal BatchNorm Fisher).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kfac_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_kfac.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)
_L = ctypes.c_long


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math) in place."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    """Load an oracle build and declare its C signatures."""
    lib = ctypes.CDLL(path)
    if lib is not None:
        lib.orc_set_threads.argtypes = [ctypes.c_int]
        lib.orc_set_threads.restype = ctypes.c_int
        lib.orc_im2col.argtypes = [_dp] + [_L] * 10 + [ctypes.c_int, _dp]
        lib.orc_gram.argtypes = [_dp, _L, _L, _dp]
        lib.orc_factor_ema.argtypes = [_dp, _dp, _L, _L, ctypes.c_double]
        lib.orc_gram_entries.argtypes = [_dp] + [_L] * 10 + [ctypes.c_int, _lp, _lp, _L, _dp]
        lib.orc_weight_grad.argtypes = [_dp, _dp, _L, _L, _L, _L, _dp]
        lib.orc_pi_damping.argtypes = [_dp, _L, _dp, _L, ctypes.c_double, ctypes.c_int, _dp, _dp]
        lib.orc_cholesky_upper.argtypes = [_dp, _L]
        lib.orc_trtri_upper.argtypes = [_dp, _L]
        lib.orc_lauum_upper.argtypes = [_dp, _L, _dp]
        lib.orc_damped_inverse.argtypes = [_dp, _L, ctypes.c_double, _dp]
        lib.orc_precondition.argtypes = [_dp, _L, _dp, _L, _dp, _dp]
        lib.orc_precondition_rows.argtypes = [_dp, _L, _dp, _L, _dp, _lp, _L, _dp]
        lib.orc_weight_update.argtypes = [_dp, _dp, _L, _L, ctypes.c_double]
        lib.orc_is_refresh_step.argtypes = [_L, _L, _L]
        lib.orc_pack_upper.argtypes = [_dp, _L, _dp]
        lib.orc_unpack_upper.argtypes = [_dp, _L, _dp]
        lib.orc_bn_diag_fisher.argtypes = [_dp, _L, _L, ctypes.c_double, ctypes.c_double,
                                           _dp, _dp, _dp]
        for f in ("orc_im2col", "orc_gram", "orc_factor_ema", "orc_gram_entries",
                  "orc_weight_grad", "orc_pi_damping", "orc_cholesky_upper",
                  "orc_trtri_upper", "orc_lauum_upper", "orc_damped_inverse",
                  "orc_precondition", "orc_precondition_rows", "orc_bn_diag_fisher",
                  "orc_weight_update", "orc_is_refresh_step", "orc_pack_upper", "orc_unpack_upper"):
            getattr(lib, f).restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


@contextlib.contextmanager
def variant(path: str):
    """Run the wrappers against another build of the oracle (used by the
    tests that plant a mistake in a copy of the C source)."""
    global _lib
    old = _load()
    _lib = _bind(path)
    try:
        yield
    finally:
        _lib = old


def _d(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def set_threads(n: int = 0) -> int:
    """Set (n > 0) and return the OpenMP thread count of the oracle."""
    return int(_load().orc_set_threads(int(n)))


def out_hw(h, w, kh, kw, sh, sw, ph, pw):
    return (h + 2 * ph - kh) // sh + 1, (w + 2 * pw - kw) // sw + 1


def im2col(x, kh=1, kw=1, stride=(1, 1), pad=(0, 0), append_one=False):
    """Patch matrix P[M, d] of NHWC input x[n, h, w, c] (see kfac_oracle.c)."""
    x = _d(x)
    if x.ndim == 2:
        x = x.reshape(x.shape[0], 1, 1, x.shape[1])
    n, h, w, c = x.shape
    ho, wo = out_hw(h, w, kh, kw, stride[0], stride[1], pad[0], pad[1])
    d = kh * kw * c + (1 if append_one else 0)
    P = np.empty((n * ho * wo, d), dtype=np.float64)
    rc = _load().orc_im2col(_p(x), n, h, w, c, kh, kw, stride[0], stride[1], pad[0], pad[1],
                            int(bool(append_one)), _p(P))
    assert rc == 0, rc
    return P


def gram(P):
    """Full symmetric P^T P (un-normalised factor statistic)."""
    P = _d(P)
    M, d = P.shape
    S = np.empty((d, d), dtype=np.float64)
    assert _load().orc_gram(_p(P), M, d, _p(S)) == 0
    return S


def factor_ema(F, P, xi):
    """F <- xi F + (1 - xi) P^T P / M, returned as a new full symmetric array."""
    F = _d(F).copy()
    P = _d(P)
    M, d = P.shape
    assert F.shape == (d, d)
    assert _load().orc_factor_ema(_p(F), _p(P), M, d, float(xi)) == 0
    return F


def gram_entries(x, ii, jj, kh=1, kw=1, stride=(1, 1), pad=(0, 0), append_one=False):
    """Entries (ii[t], jj[t]) of P^T P computed directly from x (no P)."""
    x = _d(x)
    if x.ndim == 2:
        x = x.reshape(x.shape[0], 1, 1, x.shape[1])
    n, h, w, c = x.shape
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    out = np.empty(len(ii), dtype=np.float64)
    rc = _load().orc_gram_entries(_p(x), n, h, w, c, kh, kw, stride[0], stride[1], pad[0], pad[1],
                                  int(bool(append_one)), ii.ctypes.data_as(_lp),
                                  jj.ctypes.data_as(_lp), len(ii), _p(out))
    assert rc == 0, rc
    return out


def weight_grad(P, Gam, nsamples):
    """grad[dG, dA] = Gam^T P / nsamples."""
    P = _d(P)
    Gam = _d(Gam)
    M, dA = P.shape
    dG = Gam.shape[1]
    assert Gam.shape[0] == M
    out = np.empty((dG, dA), dtype=np.float64)
    assert _load().orc_weight_grad(_p(P), _p(Gam), M, dA, dG, int(nsamples), _p(out)) == 0
    return out


def pi_damping(A, G, gamma, pi_split=True):
    """(damp_A, damp_G) for factors A, G (pi-split, or sqrt(gamma) each)."""
    A = _d(A)
    G = _d(G)
    da, dg = ctypes.c_double(), ctypes.c_double()
    assert _load().orc_pi_damping(_p(A), A.shape[0], _p(G), G.shape[0], float(gamma),
                                  int(bool(pi_split)), ctypes.byref(da), ctypes.byref(dg)) == 0
    return da.value, dg.value


def cholesky_upper(A):
    """Upper Cholesky factor U (A = U^T U); raises on a non-PD input."""
    U = _d(A).copy()
    info = _load().orc_cholesky_upper(_p(U), U.shape[0])
    if info:
        raise np.linalg.LinAlgError(f"not positive definite at pivot {info - 1}")
    return U


def trtri_upper(U):
    X = _d(U).copy()
    assert _load().orc_trtri_upper(_p(X), X.shape[0]) == 0
    return X


def lauum_upper(V):
    V = _d(V)
    out = np.empty_like(V)
    assert _load().orc_lauum_upper(_p(V), V.shape[0], _p(out)) == 0
    return out


def damped_inverse(F, damp):
    """(F + damp I)^-1 by Cholesky -> triangular inverse -> U^-1 U^-T."""
    F = _d(F)
    out = np.empty_like(F)
    info = _load().orc_damped_inverse(_p(F), F.shape[0], float(damp), _p(out))
    if info:
        raise np.linalg.LinAlgError(f"not positive definite at pivot {info - 1}")
    return out


def precondition(Ginv, grad, Ainv):
    """Ginv @ grad @ Ainv (Eq. 7 in row-major form)."""
    Ginv, grad, Ainv = _d(Ginv), _d(grad), _d(Ainv)
    dG, dA = grad.shape
    out = np.empty((dG, dA), dtype=np.float64)
    assert _load().orc_precondition(_p(Ginv), dG, _p(grad), dA, _p(Ainv), _p(out)) == 0
    return out


def precondition_rows(Ginv, grad, Ainv, rows):
    """Rows `rows` of Ginv @ grad @ Ainv, evaluated as (Ginv[rows] @ grad) @ Ainv."""
    Ginv, grad, Ainv = _d(Ginv), _d(grad), _d(Ainv)
    dG, dA = grad.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert rows.min() >= 0 and rows.max() < dG
    out = np.empty((len(rows), dA), dtype=np.float64)
    assert _load().orc_precondition_rows(_p(Ginv), dG, _p(grad), dA, _p(Ainv), rows.ctypes.data_as(_lp),
                                         len(rows), _p(out)) == 0
    return out


def weight_update(w, P, eta):
    """w - eta * P (Eq. 8), returned as a new array."""
    w = _d(w).copy()
    P = _d(P)
    assert w.shape == P.shape
    assert _load().orc_weight_update(_p(w), _p(P), w.shape[0], w.shape[1], float(eta)) == 0
    return w


def is_refresh_step(t, warmup, every):
    """True when step t of the stale-factor schedule refreshes the factors and inverses."""
    return bool(_load().orc_is_refresh_step(int(t), int(warmup), int(every)))


def pack_upper(F):
    """Packed upper triangle of F [d, d]: row i's entries j >= i, row after row."""
    F = _d(F)
    d = F.shape[0]
    out = np.empty(d * (d + 1) // 2)
    assert _load().orc_pack_upper(_p(F), d, _p(out)) == 0
    return out


def unpack_upper(Fp, d):
    """Symmetric [d, d] matrix from its packed upper triangle."""
    Fp = _d(Fp)
    assert Fp.size == d * (d + 1) // 2
    F = np.empty((d, d))
    assert _load().orc_unpack_upper(_p(Fp), d, _p(F)) == 0
    return F


def kfac_schedule(A0, G0, steps, xi, gamma, warmup, every):
    """The stale-factor schedule over a sequence of steps of one layer.
    steps: list of (P, Gam, grad) per step.  Returns the preconditioned
    gradient of every step: refresh steps update both factors (running
    average from A0, G0), damp and invert them; other steps reuse the last
    inverses."""
    A, G = _d(A0).copy(), _d(G0).copy()
    Ainv = Ginv = None
    outs = []
    for t, (P, Gam, grad) in enumerate(steps):
        if is_refresh_step(t, warmup, every) or Ainv is None:
            A = factor_ema(A, P, xi)
            G = factor_ema(G, Gam, xi)
            da, dg = pi_damping(A, G, gamma)
            Ainv = damped_inverse(A, da)
            Ginv = damped_inverse(G, dg)
        outs.append(precondition(Ginv, grad, Ainv))
    return outs


def bn_diag_fisher(x, gamma, xi=0.0, F=None):
    """(F, gmean, out) of the diagonal BatchNorm Fisher for x[ns, C]."""
    x = _d(x)
    ns, C = x.shape
    F = np.zeros(C) if F is None else _d(F).copy()
    g = np.empty(C)
    o = np.empty(C)
    assert _load().orc_bn_diag_fisher(_p(x), ns, C, float(gamma), float(xi), _p(F), _p(g), _p(o)) == 0
    return F, g, o


def kfac_layer_step(A0, G0, P, Gam, grad, xi, gamma, pi_split=True):
    """One full layer step: EMA both factors, pi-damp, invert, precondition.

    Returns a dict with the updated factors, damping values, inverses and the
    preconditioned gradient.  Convenience composition of the functions above.
    """
    A = factor_ema(A0, P, xi)
    G = factor_ema(G0, Gam, xi)
    dA_, dG_ = pi_damping(A, G, gamma, pi_split)
    Ainv = damped_inverse(A, dA_)
    Ginv = damped_inverse(G, dG_)
    out = precondition(Ginv, grad, Ainv)
    return dict(A=A, G=G, damp_A=dA_, damp_G=dG_, Ainv=Ainv, Ginv=Ginv, precond=out)
