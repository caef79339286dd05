"""Thin ctypes binding of libkfac_gb300.so (C ABI in include/kfac.h).

Argument marshalling only: every step of the K-FAC curvature path runs in the
library's CUDA kernels.  PyTorch supplies device memory (tensors, the
workspace) and the stream.  There is no CPU or PyTorch fallback: if the
library is missing, loading it raises.

The functions keep the C names:
  kfac_factor_update   (Osawa et al. section 3.2, Eq. 5 + running average)
  kfac_damp_invert     (Eq. 6, pi-split Tikhonov damping)
  kfac_precondition    (Eq. 7)
  kfac_bn_diag_fisher  (diagonal BatchNorm Fisher, section 1)
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkfac_gb300.so")

KFAC_OK, KFAC_ERR_INVALID, KFAC_ERR_UNSUPPORTED, KFAC_ERR_NOT_PD, KFAC_ERR_CUDA, KFAC_ERR_WORKSPACE = range(6)
KFAC_BF16, KFAC_F32, KFAC_F16 = 0, 1, 2
KFAC_LAYOUT_FULL, KFAC_LAYOUT_PACKED_UPPER = 0, 1
# bits of the device error word (the first int32 of a call's workspace)
ERRW_TIMEOUT_OPERAND, ERRW_TIMEOUT_STAGE, ERRW_TIMEOUT_ACCUM, ERRW_TIMEOUT_DRAIN, ERRW_NONFINITE = 1, 2, 4, 8, 16

EXPORTS = ("kfac_status_string", "kfac_version", "kfac_launch_count", "kfac_timing_enable",
           "kfac_timing_read", "kfac_timing_kind_name", "kfac_factor_update_workspace_size",
           "kfac_factor_update", "kfac_damp_invert_workspace_size", "kfac_damp_invert",
           "kfac_precondition_workspace_size", "kfac_precondition", "kfac_bn_diag_fisher",
           "kfac_noalloc_scratch_bytes", "kfac_precondition_noalloc", "kfac_timing_read_launches")


class KfacError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


class FactorDesc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("x", ctypes.c_void_p),
                ("n", ctypes.c_int32), ("h", ctypes.c_int32), ("w", ctypes.c_int32), ("c", ctypes.c_int32),
                ("kh", ctypes.c_int32), ("kw", ctypes.c_int32),
                ("stride_h", ctypes.c_int32), ("stride_w", ctypes.c_int32),
                ("pad_h", ctypes.c_int32), ("pad_w", ctypes.c_int32),
                ("append_one", ctypes.c_int32),
                ("F", ctypes.c_void_p), ("ldf", ctypes.c_int64),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("layout", ctypes.c_int32)]


class InvertDesc(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("dA", ctypes.c_int32), ("lda", ctypes.c_int64),
                ("G", ctypes.c_void_p), ("dG", ctypes.c_int32), ("ldg", ctypes.c_int64),
                ("A_inv", ctypes.c_void_p), ("ld_ainv", ctypes.c_int64),
                ("G_inv", ctypes.c_void_p), ("ld_ginv", ctypes.c_int64),
                ("A_inv_bf16", ctypes.c_void_p), ("ld_ainv_bf16", ctypes.c_int64),
                ("G_inv_bf16", ctypes.c_void_p), ("ld_ginv_bf16", ctypes.c_int64),
                ("layout_A", ctypes.c_int32), ("layout_G", ctypes.c_int32),
                ("copy_dtype", ctypes.c_int32)]


class PrecondDesc(ctypes.Structure):
    _fields_ = [("dG", ctypes.c_int32), ("dA", ctypes.c_int32),
                ("G_inv", ctypes.c_void_p), ("ld_ginv", ctypes.c_int64),
                ("A_inv", ctypes.c_void_p), ("ld_ainv", ctypes.c_int64),
                ("grad", ctypes.c_void_p), ("ld_grad", ctypes.c_int64),
                ("out", ctypes.c_void_p), ("ld_out", ctypes.c_int64),
                ("w", ctypes.c_void_p), ("ld_w", ctypes.c_int64),
                ("eta", ctypes.c_float)]


class BnDesc(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("C", ctypes.c_int32), ("F", ctypes.c_void_p),
                ("grad_mean", ctypes.c_void_p), ("precond", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load libkfac_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.kfac_status_string.argtypes = [i32]
        lib.kfac_status_string.restype = ctypes.c_char_p
        lib.kfac_version.restype = i32
        lib.kfac_launch_count.restype = ctypes.c_longlong
        lib.kfac_timing_enable.argtypes = [i32]
        lib.kfac_timing_enable.restype = i32
        lib.kfac_timing_read.argtypes = [vp, vp, i32]
        lib.kfac_timing_read.restype = i32
        lib.kfac_timing_read_launches.argtypes = [vp, vp, vp, vp, i32]
        lib.kfac_timing_read_launches.restype = i32
        lib.kfac_timing_kind_name.argtypes = [i32]
        lib.kfac_timing_kind_name.restype = ctypes.c_char_p
        lib.kfac_factor_update_workspace_size.argtypes = [vp, i32]
        lib.kfac_factor_update_workspace_size.restype = sz
        lib.kfac_factor_update.argtypes = [vp, i32, vp, sz, vp]
        lib.kfac_damp_invert_workspace_size.argtypes = [vp, i32]
        lib.kfac_damp_invert_workspace_size.restype = sz
        lib.kfac_damp_invert.argtypes = [vp, i32, f32, i32, vp, vp, vp, sz, vp]
        lib.kfac_precondition_workspace_size.argtypes = [vp, i32, i32]
        lib.kfac_precondition_workspace_size.restype = sz
        lib.kfac_precondition.argtypes = [vp, i32, i32, vp, sz, vp]
        lib.kfac_bn_diag_fisher.argtypes = [vp, i32, i32, f32, f32, vp]
        lib.kfac_noalloc_scratch_bytes.restype = sz
        lib.kfac_precondition_noalloc.argtypes = [vp, i32, i32, vp]
        for f in ("kfac_factor_update", "kfac_damp_invert", "kfac_precondition", "kfac_bn_diag_fisher",
                  "kfac_precondition_noalloc"):
            getattr(lib, f).restype = i32
        _lib = lib
    return _lib


def launch_count() -> int:
    """Kernel launches the library has enqueued in this process."""
    return int(load().kfac_launch_count())


def timing_enable(on: bool = True) -> bool:
    """Turn the library's per-kernel event timing on or off (diagnostic)."""
    return bool(load().kfac_timing_enable(int(bool(on))))


def timing_read() -> dict:
    """{kernel kind: (total ms, launches)} since the last read (synchronises)."""
    lib = load()
    n = 32
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_longlong * n)()
    _check(lib.kfac_timing_read(ms, cnt, n), "kfac_timing_read")
    out = {}
    for k in range(n):
        name = lib.kfac_timing_kind_name(k).decode()
        if name and cnt[k]:
            out[name] = (ms[k], int(cnt[k]))
    return out


def timing_read_launches(n: int = 65536) -> list:
    """[(start ms, duration ms, kernel kind name, stream id)] of every recorded
    launch in enqueue order, since the last read (synchronises); stream ids
    number the launch streams 0, 1, ... in order of first appearance."""
    lib = load()
    st = (ctypes.c_double * n)()
    du = (ctypes.c_double * n)()
    kd = (ctypes.c_int * n)()
    sm = (ctypes.c_ulonglong * n)()
    cnt = lib.kfac_timing_read_launches(st, du, kd, sm, n)
    if cnt < 0:
        raise KfacError(KFAC_ERR_CUDA, "kfac_timing_read_launches")
    ids = {}
    return [(st[i], du[i], lib.kfac_timing_kind_name(kd[i]).decode(), ids.setdefault(sm[i], len(ids)))
            for i in range(min(cnt, n))]


def status_string(status: int) -> str:
    return load().kfac_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, what: str):
    if status != KFAC_OK:
        raise KfacError(status, what)


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise KfacError(KFAC_ERR_WORKSPACE, "workspace too small")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _ld(t: torch.Tensor) -> int:
    assert t.dim() == 2 and t.stride(1) == 1, "matrices must be row-major with unit column stride"
    return t.stride(0)


# ------------------------------------------------------------ factor update

@dataclass
class FactorSource:
    """One factor update: F[:d, :d] (upper) <- beta F + alpha P^T P, P the patch
    matrix of x.  x: NHWC [n, h, w, c] (conv) or [rows, c] (FC / output grads),
    bf16, fp16 or fp32.  With packed, F is the packed upper triangle (a 1-D
    tensor of d(d+1)/2 floats, see pack_upper)."""
    x: torch.Tensor
    F: torch.Tensor
    kh: int = 1
    kw: int = 1
    stride: tuple = (1, 1)
    pad: tuple = (0, 0)
    append_one: bool = False
    alpha: float = 1.0
    beta: float = 0.0
    packed: bool = False


_DTYPES = {torch.bfloat16: KFAC_BF16, torch.float16: KFAC_F16, torch.float32: KFAC_F32}


def packed_size(d: int) -> int:
    """Floats of a packed upper triangle of order d."""
    return d * (d + 1) // 2


def pack_upper(F: torch.Tensor) -> torch.Tensor:
    """The packed upper triangle (KFAC_LAYOUT_PACKED_UPPER) of a square
    matrix: row i's entries j >= i, row after row (a layout conversion)."""
    d = F.shape[0]
    iu = torch.triu_indices(d, d, device=F.device)
    return F[iu[0], iu[1]].contiguous()


def unpack_upper(Fp: torch.Tensor, d: int) -> torch.Tensor:
    """Square matrix holding a packed upper triangle (zeros below)."""
    out = torch.zeros(d, d, dtype=Fp.dtype, device=Fp.device)
    iu = torch.triu_indices(d, d, device=Fp.device)
    out[iu[0], iu[1]] = Fp
    return out


def _fld(F: torch.Tensor, packed: bool) -> int:
    if packed:
        assert F.dim() == 1 and F.is_contiguous() and F.dtype == torch.float32
        return 0
    return _ld(F)


def _factor_descs(sources: Sequence[FactorSource]):
    arr = (FactorDesc * max(len(sources), 1))()
    for i, s in enumerate(sources):
        x = s.x
        assert x.is_contiguous(), "x must be dense"
        if x.dim() == 2:
            n, h, w, c = x.shape[0], 1, 1, x.shape[1]
        else:
            n, h, w, c = x.shape
        if x.dtype not in _DTYPES:
            raise TypeError(f"unsupported source dtype {x.dtype}")
        assert s.F.dtype == torch.float32
        arr[i] = FactorDesc(_DTYPES[x.dtype], x.data_ptr(), n, h, w, c, s.kh, s.kw, s.stride[0], s.stride[1],
                            s.pad[0], s.pad[1], int(bool(s.append_one)), s.F.data_ptr(), _fld(s.F, s.packed),
                            float(s.alpha), float(s.beta),
                            KFAC_LAYOUT_PACKED_UPPER if s.packed else KFAC_LAYOUT_FULL)
    return arr


def kfac_factor_update_workspace_size(sources: Sequence[FactorSource]) -> int:
    arr = _factor_descs(sources)
    return int(load().kfac_factor_update_workspace_size(arr, len(sources)))


def kfac_factor_update(sources: Sequence[FactorSource], workspace: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """Enqueue the factor updates; returns the workspace used (its first int32
    is the library's device error word: 0 = no timeout and no NaN or infinite
    output; ERRW_* bits otherwise)."""
    lib = load()
    arr = _factor_descs(sources)
    need = int(lib.kfac_factor_update_workspace_size(arr, len(sources)))
    if need == 0 and len(sources):
        _check(lib.kfac_factor_update(arr, len(sources), None, 0, _stream(stream)), "kfac_factor_update")
    ws = _workspace(need, sources[0].x.device if sources else "cuda", workspace)
    _check(lib.kfac_factor_update(arr, len(sources), ws.data_ptr(), ws.numel() * ws.element_size(),
                                  _stream(stream)), "kfac_factor_update")
    return ws


# ------------------------------------------------------------ damp + invert

@dataclass
class InvertPair:
    """Both factors of one layer and where their damped inverses go.  The
    optional 16-bit copies are bf16 or fp16 (both the same dtype); a packed
    factor is a 1-D tensor of d(d+1)/2 floats (then dA / dG are required)."""
    A: torch.Tensor
    G: torch.Tensor
    A_inv: torch.Tensor
    G_inv: torch.Tensor
    A_inv_bf16: Optional[torch.Tensor] = None
    G_inv_bf16: Optional[torch.Tensor] = None
    dA: Optional[int] = None
    dG: Optional[int] = None
    packed_A: bool = False
    packed_G: bool = False


def _invert_descs(pairs: Sequence[InvertPair]):
    arr = (InvertDesc * max(len(pairs), 1))()
    for i, p in enumerate(pairs):
        dA = p.dA or p.A_inv.shape[0]
        dG = p.dG or p.G_inv.shape[0]
        copies = {t.dtype for t in (p.A_inv_bf16, p.G_inv_bf16) if t is not None}
        if not copies <= {torch.bfloat16, torch.float16} or len(copies) > 1:
            raise TypeError(f"16-bit inverse copies must be both bf16 or both fp16, got {copies}")
        cdt = KFAC_F16 if copies == {torch.float16} else KFAC_BF16
        arr[i] = InvertDesc(p.A.data_ptr(), dA, _fld(p.A, p.packed_A), p.G.data_ptr(), dG, _fld(p.G, p.packed_G),
                            p.A_inv.data_ptr(), _ld(p.A_inv), p.G_inv.data_ptr(), _ld(p.G_inv),
                            _ptr(p.A_inv_bf16), _ld(p.A_inv_bf16) if p.A_inv_bf16 is not None else 0,
                            _ptr(p.G_inv_bf16), _ld(p.G_inv_bf16) if p.G_inv_bf16 is not None else 0,
                            KFAC_LAYOUT_PACKED_UPPER if p.packed_A else KFAC_LAYOUT_FULL,
                            KFAC_LAYOUT_PACKED_UPPER if p.packed_G else KFAC_LAYOUT_FULL, cdt)
    return arr


def kfac_damp_invert_workspace_size(pairs: Sequence[InvertPair]) -> int:
    return int(load().kfac_damp_invert_workspace_size(_invert_descs(pairs), len(pairs)))


def kfac_damp_invert(pairs: Sequence[InvertPair], gamma: float, pi_split: bool = True,
                     info: Optional[torch.Tensor] = None, damp: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Enqueue the damped inversions; returns the workspace used (its first
    int32 is the library's device error word: 0 = no timeout and no NaN or
    infinite output; ERRW_* bits otherwise)."""
    lib = load()
    arr = _invert_descs(pairs)
    need = int(lib.kfac_damp_invert_workspace_size(arr, len(pairs)))
    ws = _workspace(need, pairs[0].A.device if pairs else "cuda", workspace)
    if info is not None:
        assert info.dtype == torch.int32 and info.numel() >= 2 * len(pairs)
    if damp is not None:
        assert damp.dtype == torch.float32 and damp.numel() >= 2 * len(pairs)
    _check(lib.kfac_damp_invert(arr, len(pairs), float(gamma), int(bool(pi_split)), _ptr(info), _ptr(damp),
                                ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "kfac_damp_invert")
    return ws


# ------------------------------------------------------------ precondition

@dataclass
class PrecondItem:
    """out = G_inv @ grad @ A_inv for one layer (grad [dG, dA]); with w, also
    w -= eta * out in place (out may then be None)."""
    G_inv: torch.Tensor
    A_inv: torch.Tensor
    grad: torch.Tensor
    out: Optional[torch.Tensor]
    dG: Optional[int] = None
    dA: Optional[int] = None
    w: Optional[torch.Tensor] = None
    eta: float = 0.0


def _precond_descs(items: Sequence[PrecondItem]):
    arr = (PrecondDesc * max(len(items), 1))()
    for i, it in enumerate(items):
        dG = it.dG or it.grad.shape[0]
        dA = it.dA or it.grad.shape[1]
        if it.w is not None and it.w.dtype != torch.float32:
            raise TypeError("w must be fp32")
        arr[i] = PrecondDesc(dG, dA, it.G_inv.data_ptr(), _ld(it.G_inv), it.A_inv.data_ptr(), _ld(it.A_inv),
                             it.grad.data_ptr(), _ld(it.grad),
                             it.out.data_ptr() if it.out is not None else None,
                             _ld(it.out) if it.out is not None else 0,
                             it.w.data_ptr() if it.w is not None else None,
                             _ld(it.w) if it.w is not None else 0, float(it.eta))
    return arr


def _precond_dtype(items: Sequence[PrecondItem]) -> int:
    dts = {it.grad.dtype for it in items} | {it.A_inv.dtype for it in items} | {it.G_inv.dtype for it in items}
    if len(dts) == 1 and next(iter(dts)) in _DTYPES:
        return _DTYPES[next(iter(dts))]
    raise TypeError(f"operands must be all bf16, all fp16 or all fp32, got {dts}")


def kfac_precondition_workspace_size(items: Sequence[PrecondItem]) -> int:
    return int(load().kfac_precondition_workspace_size(_precond_descs(items), len(items),
                                                       _precond_dtype(items)))


def kfac_precondition(items: Sequence[PrecondItem], workspace: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    lib = load()
    arr = _precond_descs(items)
    dt = _precond_dtype(items)
    need = int(lib.kfac_precondition_workspace_size(arr, len(items), dt))
    ws = _workspace(need, items[0].grad.device if items else "cuda", workspace)
    _check(lib.kfac_precondition(arr, len(items), dt, ws.data_ptr(), ws.numel() * ws.element_size(),
                                 _stream(stream)), "kfac_precondition")
    return ws


def kfac_precondition_noalloc(items: Sequence[PrecondItem], stream=None) -> None:
    """kfac_precondition with the library's fixed device scratch instead of a
    workspace: for callers that cannot allocate device memory (see kfac.h)."""
    lib = load()
    arr = _precond_descs(items)
    _check(lib.kfac_precondition_noalloc(arr, len(items), _precond_dtype(items), _stream(stream)),
           "kfac_precondition_noalloc")


# ------------------------------------------------------------ BN diagonal Fisher

@dataclass
class BnItem:
    x: torch.Tensor            # [n_samples, C] fp32
    F: torch.Tensor            # [C] fp32
    precond: torch.Tensor      # [C] fp32
    grad_mean: Optional[torch.Tensor] = None


def kfac_bn_diag_fisher(items: Sequence[BnItem], gamma: float, xi: float = 0.0, stream=None) -> None:
    lib = load()
    arr = (BnDesc * max(len(items), 1))()
    ns = items[0].x.shape[0] if items else 1
    for i, it in enumerate(items):
        assert it.x.dtype == torch.float32 and it.x.is_contiguous() and it.x.shape[0] == ns
        arr[i] = BnDesc(it.x.data_ptr(), it.x.shape[1], it.F.data_ptr(), _ptr(it.grad_mean),
                        it.precond.data_ptr())
    _check(lib.kfac_bn_diag_fisher(arr, len(items), ns, float(gamma), float(xi), _stream(stream)),
           "kfac_bn_diag_fisher")
