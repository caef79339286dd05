"""Seeded synthetic inputs and layer shapes for the K-FAC curvature step.

This module holds shapes and random draws only -- none of the method's
arithmetic -- so that the CUDA path and the CPU oracle can be fed the same
inputs.  Tensors are drawn on the host with numpy's PCG64 generator from a
seed derived from (workload, layer, tensor kind) and rounded to bf16 by
round-to-nearest-even.

Shapes follow the ResNet-50 set-up used by Osawa et al., "Large-Scale
Distributed Second-Order Optimization Using Kronecker-Factored Approximate
Curvature for Deep Convolutional Neural Networks" (section 2: 32 samples per
GPU; Tables 1-2: ResNet-50 on ImageNet).  ImageNet itself is replaced by
these synthetic tensors with the same shapes:
  activations  = ReLU(N(0, 1))          (bf16, NHWC)
  output grads = N(0, 1e-3^2)           (bf16, rows [M, C_out])
  weight grads = N(0, 1e-3^2)           (bf16, [C_out, kh*kw*C_in (+1)])
  BN grads     = N(0, 1e-2^2)           (fp32, per-sample [N, C])
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Layer:
    """One K-FAC layer: a convolution (or FC when k == 1 and hin == 1)."""
    name: str
    cin: int
    cout: int
    k: int
    stride: int
    pad: int
    hin: int     # input spatial size (square)
    hout: int    # output spatial size (square)
    bias: bool = False

    @property
    def d_a(self) -> int:
        return self.k * self.k * self.cin + (1 if self.bias else 0)

    @property
    def d_g(self) -> int:
        return self.cout

    def rows(self, batch: int) -> int:
        return batch * self.hout * self.hout


def resnet50_layers() -> list[Layer]:
    """The 54 weight layers of ResNet-50 (v1: stride on the first 1x1 of a
    down-sampling block), in forward order, for a 224x224 input."""
    L = [Layer("conv1", 3, 64, 7, 2, 3, 224, 112)]
    spec = [(3, 64, 256, 56, 56), (4, 128, 512, 56, 28), (6, 256, 1024, 28, 14),
            (3, 512, 2048, 14, 7)]
    cin = 64
    for si, (nblocks, width, cout, hin, hout) in enumerate(spec):
        for b in range(nblocks):
            s = 1 if (b > 0 or si == 0) else 2
            h_in = hin if b == 0 else hout
            p = f"s{si + 1}b{b + 1}"
            L.append(Layer(p + "_1x1a", cin, width, 1, s, 0, h_in, hout))
            L.append(Layer(p + "_3x3", width, width, 3, 1, 1, hout, hout))
            L.append(Layer(p + "_1x1b", width, cout, 1, 1, 0, hout, hout))
            if b == 0:
                L.append(Layer(p + "_proj", cin, cout, 1, s, 0, h_in, hout))
            cin = cout
    L.append(Layer("fc", 2048, 1000, 1, 1, 0, 1, 1, bias=True))
    return L


def resnet50_bn_channels() -> list[int]:
    """Channel count of each of ResNet-50's 53 BatchNorm layers (one after
    every convolution)."""
    return [l.cout for l in resnet50_layers() if l.name != "fc"]


# ------------------------------------------------------------------ drawing

def seed_of(*parts) -> int:
    """Stable 63-bit seed from a tuple of labels."""
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _rng(*parts) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_of(*parts)))


def normal_f32(shape, std, *parts) -> np.ndarray:
    return (_rng(*parts).standard_normal(size=shape, dtype=np.float32) * np.float32(std))


def relu_normal_f32(shape, *parts) -> np.ndarray:
    x = _rng(*parts).standard_normal(size=shape, dtype=np.float32)
    np.maximum(x, 0.0, out=x)
    return x


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """Round an fp32 array to bf16 (round to nearest even), on the host."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def layer_inputs(layer: Layer, batch: int, *tag, grad_w: bool = True):
    """Host bf16 tensors (x NHWC, g [M, C_out], grad [d_G, d_A]) of one layer."""
    x = to_bf16(relu_normal_f32((batch, layer.hin, layer.hin, layer.cin), *tag, layer.name, "x"))
    g = to_bf16(normal_f32((layer.rows(batch), layer.cout), 1e-3, *tag, layer.name, "g"))
    w = to_bf16(normal_f32((layer.d_g, layer.d_a), 1e-3, *tag, layer.name, "gradW")) if grad_w else None
    return x, g, w


def bn_grads(channels: list[int], nsamples: int, *tag):
    """Per-sample BN gradients for the scale and shift of every BN layer:
    a list of (x_gamma, x_beta) fp32 host arrays of shape [nsamples, C]."""
    return [(normal_f32((nsamples, c), 1e-2, *tag, i, "bn_gamma"),
             normal_f32((nsamples, c), 1e-2, *tag, i, "bn_beta")) for i, c in enumerate(channels)]


# ------------------------------------------------------------- small cases

def fc_small_fp32(tag="fc64x32"):
    """The single-FC-layer case in fp32: a[32, 64] = ReLU(N(0,1)),
    g[32, 32] ~ N(0, 0.01^2).  The bias column is appended by the method."""
    a = relu_normal_f32((32, 64), tag, "a")
    g = normal_f32((32, 32), 1e-2, tag, "g")
    return a, g


def conv_3x3_256(batch=32):
    """The single ResNet-50-style 3x3 convolution: Cin = Cout = 256, 14x14,
    stride 1, pad 1, no bias."""
    return Layer("conv3x3_256", 256, 256, 3, 1, 1, 14, 14)


def fc_4096():
    """Dense-contraction stress layer: FC 4096 -> 4096 with bias, 8192 rows."""
    return Layer("fc4096", 4096, 4096, 1, 1, 0, 1, 1, bias=True)
