"""Seeded synthetic inputs for dgrad, shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method: shapes are listed explicitly
(grad_out's spatial size included) and tensors come from
``torch.Generator('cpu').manual_seed(seed)`` in a fixed order (grad_out first,
then weight), as fp32 on the CPU.  Callers move them to the GPU themselves, so
the CUDA path and the CPU oracle see bit-identical inputs.

Distributions:
  * ``"uniform"``: grad_out and weight ~ U(-1, 1).
  * ``"kaiming"``: grad_out ~ N(0, 1); weight ~ N(0, 2 / (Ci * kH * kW))
    (Kaiming-normal fan-in scaling for every configuration).

The five named workloads are ResNet-shaped stand-ins for real backward passes;
no dataset is involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    Ci: int
    Co: int
    H: int
    W: int
    kH: int
    kW: int
    stride: int
    pad_h: int
    pad_w: int
    oH: int  # grad_out spatial size, listed (not derived) so this module stays arithmetic-free
    oW: int
    dist: str

    @property
    def go_shape(self):
        return (self.N, self.Co, self.oH, self.oW)

    @property
    def w_shape(self):
        return (self.Co, self.Ci, self.kH, self.kW)

    @property
    def gi_shape(self):
        return (self.N, self.Ci, self.H, self.W)

    def plan_args(self):
        return (self.N, self.Ci, self.H, self.W, self.Co, self.kH, self.kW,
                self.stride, self.pad_h, self.pad_w)

    def as_dict(self):
        return asdict(self)


WORKLOADS = {
    "tiny": Workload("tiny", 2, 3, 4, 8, 8, 3, 3, 1, 1, 1, 8, 8, "uniform"),
    "resnet_stage": Workload("resnet_stage", 32, 64, 64, 56, 56, 3, 3, 1, 1, 1, 56, 56, "kaiming"),
    "strided_downsample": Workload("strided_downsample", 32, 128, 256, 28, 28, 3, 3, 2, 1, 1, 14, 14, "kaiming"),
    "pointwise": Workload("pointwise", 64, 256, 1024, 14, 14, 1, 1, 1, 0, 0, 14, 14, "kaiming"),
    "stem": Workload("stem", 32, 3, 64, 224, 224, 7, 7, 2, 3, 3, 112, 112, "kaiming"),
}
ORDER = ["tiny", "resnet_stage", "strided_downsample", "pointwise", "stem"]


def make_tensors(go_shape, w_shape, seed: int, dist: str = "kaiming"):
    """Return (grad_out, weight) as contiguous fp32 CPU tensors drawn from ``seed``."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    if dist == "uniform":
        go = torch.rand(go_shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
        w = torch.rand(w_shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "kaiming":
        go = torch.randn(go_shape, generator=g, dtype=torch.float32)
        fan_in = w_shape[1] * w_shape[2] * w_shape[3]
        w = torch.randn(w_shape, generator=g, dtype=torch.float32) * math.sqrt(2.0 / fan_in)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return go.contiguous(), w.contiguous()


def make_inputs(wl: Workload | str, seed: int = 0):
    """Seeded (grad_out, weight) for a named workload."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    return make_tensors(wl.go_shape, wl.w_shape, seed, wl.dist)


def useful_flops(wl: Workload) -> int:
    """2 * N * Co * oH * oW * Ci * kH * kW: every (output, tap) pair, padded taps included."""
    return 2 * wl.N * wl.Co * wl.oH * wl.oW * wl.Ci * wl.kH * wl.kW


def algorithmic_bytes(wl: Workload) -> int:
    """Compulsory HBM traffic: read grad_out and weight once, write grad_input once (fp32)."""
    return 4 * (wl.N * wl.Co * wl.oH * wl.oW + wl.Co * wl.Ci * wl.kH * wl.kW
                + wl.N * wl.Ci * wl.H * wl.W)
