"""The C ABI (CPU-only checks): the library loads, exports every function
include/kfac.h declares, and rejects invalid arguments before enqueuing any
work (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

from second_order_optimisation_gb300 import kfac

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(kfac_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return kfac.load()


def test_every_declared_function_is_exported(lib):
    names = _header_functions()
    assert {"kfac_factor_update", "kfac_damp_invert", "kfac_precondition",
            "kfac_bn_diag_fisher"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(kfac.EXPORTS) <= set(names)


def test_status_strings(lib):
    for s in range(6):
        assert kfac.status_string(s).startswith("KFAC_")
    assert "unknown" in kfac.status_string(99)
    assert lib.kfac_version() >= 100


def _fdesc(**kw):
    d = dict(dtype=kfac.KFAC_BF16, x=0x1000, n=4, h=6, w=6, c=64, kh=3, kw=3, stride_h=1, stride_w=1,
             pad_h=1, pad_w=1, append_one=0, F=0x2000, ldf=576, alpha=1.0, beta=0.0)
    d.update(kw)
    return kfac.FactorDesc(**d)


@pytest.mark.parametrize("bad", [dict(x=None), dict(F=None), dict(n=0), dict(c=-1), dict(kh=0),
                                 dict(stride_w=0), dict(pad_h=-1), dict(ldf=575), dict(dtype=7),
                                 dict(h=1, w=1, kh=3, kw=3, pad_h=0, pad_w=0),
                                 dict(alpha=float("nan"))])
def test_factor_update_rejects_invalid(lib, bad):
    arr = (kfac.FactorDesc * 1)(_fdesc(**bad))
    assert lib.kfac_factor_update(arr, 1, None, 0, None) == kfac.KFAC_ERR_INVALID
    assert lib.kfac_factor_update_workspace_size(arr, 1) == 0


def test_factor_update_implicit_im2col_needs_no_patch_matrix(lib):
    # c = 64 fills whole 64-channel taps: the SYRK reads the input through an
    # im2col tensor map and no patch matrix is laid out
    arr = (kfac.FactorDesc * 1)(_fdesc())
    assert 0 < lib.kfac_factor_update_workspace_size(arr, 1) < 4 * 6 * 6 * 576 * 2


def test_factor_update_workspace_and_count_checks(lib):
    arr = (kfac.FactorDesc * 1)(_fdesc(c=8, ldf=72))
    need = lib.kfac_factor_update_workspace_size(arr, 1)
    # c = 8: the patch matrix of 4*6*6 rows x 72 bf16 columns must fit in the workspace
    assert need >= 4 * 6 * 6 * 72 * 2
    assert lib.kfac_factor_update(arr, 1, None, 0, None) == kfac.KFAC_ERR_WORKSPACE
    assert lib.kfac_factor_update(arr, 1, 0x1001, need, None) == kfac.KFAC_ERR_WORKSPACE  # misaligned
    assert lib.kfac_factor_update(arr, 1, 0x100000, need - 1024, None) == kfac.KFAC_ERR_WORKSPACE
    assert lib.kfac_factor_update(arr, -1, None, 0, None) == kfac.KFAC_ERR_INVALID
    assert lib.kfac_factor_update(None, 2, None, 0, None) == kfac.KFAC_ERR_INVALID
    assert lib.kfac_factor_update(None, 0, None, 0, None) == kfac.KFAC_OK
    # a bias column on a convolution source is not supported
    arr = (kfac.FactorDesc * 1)(_fdesc(append_one=1, ldf=577))
    assert lib.kfac_factor_update(arr, 1, 0x100000, 1 << 30, None) == kfac.KFAC_ERR_UNSUPPORTED


def _idesc(**kw):
    d = dict(A=0x1000, dA=10, lda=10, G=0x2000, dG=4, ldg=4, A_inv=0x3000, ld_ainv=10, G_inv=0x4000,
             ld_ginv=4, A_inv_bf16=None, ld_ainv_bf16=0, G_inv_bf16=None, ld_ginv_bf16=0)
    d.update(kw)
    return kfac.InvertDesc(**d)


@pytest.mark.parametrize("bad", [dict(A=None), dict(G_inv=None), dict(dA=0), dict(lda=9),
                                 dict(ld_ginv=3), dict(A_inv_bf16=0x5000, ld_ainv_bf16=9)])
def test_damp_invert_rejects_invalid(lib, bad):
    arr = (kfac.InvertDesc * 1)(_idesc(**bad))
    assert lib.kfac_damp_invert(arr, 1, 1e-3, 1, None, None, None, 0, None) == kfac.KFAC_ERR_INVALID


def test_damp_invert_unsupported_and_gamma(lib):
    arr = (kfac.InvertDesc * 1)(_idesc(A_inv_bf16=0x5000, ld_ainv_bf16=12))   # ld not a multiple of 8
    assert lib.kfac_damp_invert(arr, 1, 1e-3, 1, None, None, 0x100000, 1 << 20, None) == \
        kfac.KFAC_ERR_UNSUPPORTED
    arr = (kfac.InvertDesc * 1)(_idesc())
    assert lib.kfac_damp_invert(arr, 1, -1.0, 1, None, None, None, 0, None) == kfac.KFAC_ERR_INVALID
    assert lib.kfac_damp_invert(arr, 1, float("inf"), 1, None, None, None, 0, None) == kfac.KFAC_ERR_INVALID
    assert lib.kfac_damp_invert(arr, 1, 1e-3, 1, None, None, None, 0, None) == kfac.KFAC_ERR_WORKSPACE


def _pdesc(**kw):
    d = dict(dG=16, dA=24, G_inv=0x1000, ld_ginv=16, A_inv=0x2000, ld_ainv=24, grad=0x3000, ld_grad=24,
             out=0x4000, ld_out=24)
    d.update(kw)
    return kfac.PrecondDesc(**d)


@pytest.mark.parametrize("bad", [dict(out=None), dict(dG=0), dict(ld_grad=23), dict(ld_ainv=8)])
def test_precondition_rejects_invalid(lib, bad):
    arr = (kfac.PrecondDesc * 1)(_pdesc(**bad))
    assert lib.kfac_precondition(arr, 1, kfac.KFAC_F32, None, 0, None) == kfac.KFAC_ERR_INVALID


def test_precondition_bf16_alignment(lib):
    arr = (kfac.PrecondDesc * 1)(_pdesc(ld_grad=26, ld_out=26))
    assert lib.kfac_precondition(arr, 1, kfac.KFAC_BF16, 0x100000, 1 << 20, None) == \
        kfac.KFAC_ERR_UNSUPPORTED
    assert lib.kfac_precondition(arr, 1, 5, 0x100000, 1 << 20, None) == kfac.KFAC_ERR_INVALID


def test_bn_rejects_invalid(lib):
    d = kfac.BnDesc(0x1000, 64, 0x2000, None, 0x3000)
    arr = (kfac.BnDesc * 1)(d)
    assert lib.kfac_bn_diag_fisher(arr, 1, 0, 1e-3, 0.0, None) == kfac.KFAC_ERR_INVALID
    assert lib.kfac_bn_diag_fisher(arr, 1, 8, -1.0, 0.0, None) == kfac.KFAC_ERR_INVALID
    assert lib.kfac_bn_diag_fisher(arr, 1, 8, 1e-3, 1.5, None) == kfac.KFAC_ERR_INVALID
    bad = (kfac.BnDesc * 1)(kfac.BnDesc(None, 64, 0x2000, None, 0x3000))
    assert lib.kfac_bn_diag_fisher(bad, 1, 8, 1e-3, 0.0, None) == kfac.KFAC_ERR_INVALID
    assert lib.kfac_bn_diag_fisher(None, 0, 8, 1e-3, 0.0, None) == kfac.KFAC_OK


def test_product_path_has_no_fallback():
    """The binding never imports the oracle and fails loudly without the .so."""
    src = open(os.path.join(ROOT, "second_order_optimisation_gb300", "kfac.py")).read()
    assert "oracle" not in src.replace("no CPU or PyTorch fallback", "")
    for fn in os.listdir(os.path.join(ROOT, "second_order_optimisation_gb300", "csrc")):
        assert "oracle" not in open(os.path.join(ROOT, "second_order_optimisation_gb300", "csrc", fn)).read()


def test_host_memory_operands_are_rejected(lib):
    """Operands must be memory of the current device: host arrays give
    KFAC_ERR_INVALID once every other check has passed (on a machine without
    a GPU no pointer is device memory)."""
    import numpy as np
    x = np.zeros(4 * 6 * 6 * 64, dtype=np.uint16)
    F = np.zeros(576 * 576, dtype=np.float32)
    arr = (kfac.FactorDesc * 1)(_fdesc(x=x.ctypes.data, F=F.ctypes.data))
    need = lib.kfac_factor_update_workspace_size(arr, 1)
    assert need > 0
    assert lib.kfac_factor_update(arr, 1, 0x100000, need, None) == kfac.KFAC_ERR_INVALID
    g = np.zeros(16 * 24, dtype=np.float32)
    parr = (kfac.PrecondDesc * 1)(_pdesc(G_inv=g.ctypes.data, A_inv=g.ctypes.data, grad=g.ctypes.data,
                                         out=g.ctypes.data))
    assert lib.kfac_precondition(parr, 1, kfac.KFAC_F32, 0x100000, 1 << 20, None) == kfac.KFAC_ERR_INVALID
    b = kfac.BnDesc(g.ctypes.data, 16, g.ctypes.data, None, g.ctypes.data)
    assert lib.kfac_bn_diag_fisher((kfac.BnDesc * 1)(b), 1, 8, 1e-3, 0.0, None) == kfac.KFAC_ERR_INVALID
