"""Synthetic workloads: layer shapes and input recipes (no convolution arithmetic).

The shapes stand in for the workloads the pages time:
  * "pr1"        -- the smallest MobileNet-style layer of "Spatial Depthwise
                    Convolution on the GPU #3057" (N=1, C=32, 28x28, 3x3);
  * "mobilenet"  -- the MobileNet layer table of that PR at batch 64
                    (3x3, pad 1, stride 1 or 2), fp32;
  * "largek"     -- the MegEngine large-kernel depthwise article's setting
                    (section "Running time": batch 64, 384 channels) with
                    square kernels 7..31 on 32/48/64 inputs, fp32 and fp16;
  * "multidil"   -- the DynamicConvolutionOperator's fused dilation 1/3/5
                    branches (dim 64, resolution 256, batch 2), bf16,
                    stored into one concatenated output;
  * "multiplier" -- a depth-multiplier-2 5x5 training layer with bias, bf16;
  * "infer"      -- the MobileNet layer table as an inference forward in
                    channels-last layout with a fused per-channel scale,
                    shift and ReLU6 (a folded batch norm and activation),
                    fp32 and bf16.
No public dataset is involved: every tensor is drawn by ``synth`` with seed 0
and per-tensor streams. Variances are read as variances: N(0, 1/9) has
standard deviation 1/3.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

from . import synth


@dataclass
class Layer:
    N: int
    C: int
    H: int
    W: int
    k: int = 3
    s: int = 1
    p: int = 1
    d: int = 1
    m: int = 1
    bias: bool = False
    dtype: str = "f32"
    x_dist: str = "uniform"   # "uniform" = U[-1, 1], "normal" = N(0, 1)
    w_std: float | None = None  # default 1/k
    b_std: float = math.sqrt(0.1)
    name: str = ""

    @property
    def OC(self):
        return self.C * self.m

    @property
    def Ho(self):
        return (self.H + 2 * self.p - self.d * (self.k - 1) - 1) // self.s + 1

    @property
    def Wo(self):
        return (self.W + 2 * self.p - self.d * (self.k - 1) - 1) // self.s + 1

    def desc_kwargs(self):
        return dict(N=self.N, C=self.C, H=self.H, W=self.W, kernel=self.k, stride=self.s,
                    pad=self.p, dilation=self.d, multiplier=self.m, dtype=self.dtype)

    def label(self):
        return self.name or (f"N{self.N}C{self.C}H{self.H}k{self.k}s{self.s}d{self.d}"
                             f"m{self.m}{'b' if self.bias else ''}_{self.dtype}")


@dataclass
class Multi:
    """Several branches over one input writing one concatenated output."""
    N: int
    C: int
    H: int
    W: int
    dilations: tuple = (1, 3, 5)
    k: int = 3
    dtype: str = "bf16"
    x_dist: str = "normal"
    w_std: float = 1.0 / 3.0
    name: str = "multidil"

    def branches(self):
        nb = len(self.dilations)
        return [Layer(N=self.N, C=self.C, H=self.H, W=self.W, k=self.k, s=1, p=d * (self.k // 2),
                      d=d, dtype=self.dtype, x_dist=self.x_dist, w_std=self.w_std)
                for d in self.dilations], nb * self.C

    def label(self):
        return self.name


def mobilenet(N=64):
    layers = [(64, 112, 2), (128, 56, 1), (128, 56, 2), (256, 28, 1), (256, 28, 2),
              (512, 14, 1), (512, 14, 2), (1024, 7, 2)]
    return [Layer(N=N, C=c, H=h, W=h, k=3, s=s, p=1, name=f"mb_C{c}_H{h}_s{s}") for c, h, s in layers]


@dataclass
class InferLayer(Layer):
    """A forward-only layer: channels-last (NHWC) input and output, with the
    fused per-channel scale / shift / activation epilogue."""
    layout: str = "nhwc"
    act: str = "relu6"


def mobilenet_infer(N=64, dtypes=("f32", "bf16")):
    layers = [(64, 112, 2), (128, 56, 1), (128, 56, 2), (256, 28, 1), (256, 28, 2),
              (512, 14, 1), (512, 14, 2), (1024, 7, 2)]
    return [InferLayer(N=N, C=c, H=h, W=h, k=3, s=s, p=1, dtype=dt, name=f"mbi_C{c}_H{h}_s{s}_{dt}")
            for dt in dtypes for c, h, s in layers]


@dataclass
class SepLayer(InferLayer):
    """A depthwise-separable block (inference, channels-last): the depthwise
    layer with its scale / shift / activation, then a 1x1 layer to `cout`
    channels with its own scale / shift / activation."""
    cout: int = 0


def mobilenet_separable(N=64, dtype="bf16"):
    """The MobileNet layer table as depthwise-separable blocks: each 1x1 layer
    outputs the input channels of the table's next row (the last keeps 1024),
    MobileNet v1's channel sequence."""
    layers = [(64, 112, 2), (128, 56, 1), (128, 56, 2), (256, 28, 1), (256, 28, 2),
              (512, 14, 1), (512, 14, 2), (1024, 7, 2)]
    outs = [c for c, _, _ in layers[1:]] + [1024]
    return [SepLayer(N=N, C=c, H=h, W=h, k=3, s=s, p=1, dtype=dtype, cout=co, name=f"sep_C{c}_H{h}_s{s}_o{co}")
            for (c, h, s), co in zip(layers, outs)]


def pr1():
    return [Layer(N=1, C=32, H=28, W=28, k=3, s=1, p=1, name="pr1_C32_H28")]


def largek(N=64, C=384, sizes=(32, 48, 64), ks=(7, 13, 21, 27, 31), dtypes=("f32", "f16")):
    return [Layer(N=N, C=C, H=h, W=h, k=k, s=1, p=k // 2, dtype=dt, name=f"lk_H{h}_k{k}_{dt}")
            for dt in dtypes for h in sizes for k in ks]


@dataclass
class CachedLayer(Layer):
    """A forward-only large-kernel layer whose filter is fixed across calls
    (inference): served from a filter cache built once ahead of the calls
    where the shape has a cached form, else by the uncached forward."""
    cached: bool = True


def largek_infer(N=64, C=384, sizes=(32, 48, 64), ks=(13, 21, 27, 31), dtype="f16"):
    return [CachedLayer(N=N, C=C, H=h, W=h, k=k, s=1, p=k // 2, dtype=dtype, name=f"lki_H{h}_k{k}_{dtype}")
            for h in sizes for k in ks]


def multidil(N=2, C=64, H=256):
    return Multi(N=N, C=C, H=H, W=H)


def multiplier(N=128):
    return [Layer(N=N, C=256, H=28, W=28, k=5, s=1, p=2, m=2, bias=True, dtype="bf16",
                  x_dist="normal", w_std=1.0 / 5.0, name="mult_C256_H28_k5_m2")]


@dataclass
class Inputs:
    x: synth.Tensor
    w: synth.Tensor
    b: synth.Tensor | None
    gy: synth.Tensor
    extra: dict = field(default_factory=dict)


def make_x(L: Layer, seed: int = 0) -> synth.Tensor:
    xs = (L.N, L.C, L.H, L.W)
    if L.x_dist == "uniform":
        return synth.uniform_tensor(xs, L.dtype, seed, synth.STREAM_X)
    return synth.normal_tensor(xs, L.dtype, seed, synth.STREAM_X)


def make_w(L: Layer, seed: int = 0, branch: int = 0) -> synth.Tensor:
    w_std = L.w_std if L.w_std is not None else 1.0 / L.k
    return synth.normal_tensor((L.OC, L.k, L.k), L.dtype, seed, synth.STREAM_W + 16 * branch, std=w_std)


def make_b(L: Layer, seed: int = 0, branch: int = 0) -> synth.Tensor:
    return synth.normal_tensor((L.OC,), L.dtype, seed, synth.STREAM_B + 16 * branch, std=L.b_std)


def make_gy(L: Layer, seed: int = 0, gy_channels: int | None = None) -> synth.Tensor:
    gc = L.OC if gy_channels is None else gy_channels
    return synth.normal_tensor((L.N, gc, L.Ho, L.Wo), L.dtype, seed, synth.STREAM_GY)


def make_scale_shift(L: Layer, seed: int = 0):
    """Epilogue scale ~ U[0.5, 1.5] and shift ~ N(0, 0.25), one per output channel."""
    return (synth.uniform_tensor((L.OC,), L.dtype, seed, synth.STREAM_SCALE, lo=0.5, hi=1.5),
            synth.normal_tensor((L.OC,), L.dtype, seed, synth.STREAM_SHIFT, std=0.5))


def make_pointwise(L: Layer, cout: int, seed: int = 0):
    """1x1 weights [cout, C*m] ~ N(0, 1/(C*m)), scale ~ U[0.5, 1.5], shift ~ N(0, 0.25)."""
    return (synth.normal_tensor((cout, L.OC), L.dtype, seed, synth.STREAM_PW, std=1.0 / math.sqrt(L.OC)),
            synth.uniform_tensor((cout,), L.dtype, seed, synth.STREAM_PW_SCALE, lo=0.5, hi=1.5),
            synth.normal_tensor((cout,), L.dtype, seed, synth.STREAM_PW_SHIFT, std=0.5))


def make_inputs(L: Layer, seed: int = 0, branch: int = 0, gy_channels: int | None = None) -> Inputs:
    """x, w, bias and grad_out for one layer, drawn as the module docstring says."""
    return Inputs(make_x(L, seed), make_w(L, seed, branch), make_b(L, seed, branch) if L.bias else None,
                  make_gy(L, seed, gy_channels))
