"""Workload shapes and seeded synthetic inputs.

This module holds shapes and random-number draws only -- none of the
convolution's arithmetic.  Both the CUDA path's tests/bench and the CPU oracle
take their inputs from here, so the two sides see bit-identical values.

Inputs are drawn on the CPU in fp32 with a ``torch.Generator`` seeded with
``1000*workload_id + t`` (t = 0 for x, 1 for w, 2 for dy).  bf16 workloads
round the fp32 draws to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Conv2dProblem:
    """The descriptor integers of one convolution, in the order the SystemDS
    cuDNN wrapper passes them: N, C, H, W, K, R, S, pad_h, pad_w, stride_h,
    stride_w, P, Q (P and Q derived with floor division)."""

    N: int
    C: int
    H: int
    W: int
    K: int
    R: int
    S: int
    pad_h: int = 0
    pad_w: int = 0
    stride_h: int = 1
    stride_w: int = 1
    dtype: str = "f32"  # "f32" (TF32 tensor cores) or "bf16"

    @property
    def P(self) -> int:
        return (self.H + 2 * self.pad_h - self.R) // self.stride_h + 1

    @property
    def Q(self) -> int:
        return (self.W + 2 * self.pad_w - self.S) // self.stride_w + 1

    def dims(self):
        return (self.N, self.C, self.H, self.W, self.K, self.R, self.S,
                self.pad_h, self.pad_w, self.stride_h, self.stride_w, self.P, self.Q)

    @property
    def x_shape(self):
        return (self.N, self.C, self.H, self.W)

    @property
    def w_shape(self):
        return (self.K, self.C, self.R, self.S)

    @property
    def y_shape(self):
        return (self.N, self.K, self.P, self.Q)

    def flops(self) -> int:
        """Algorithmic FLOP of any one of the three ops: 2*N*K*P*Q*C*R*S."""
        return 2 * self.N * self.K * self.P * self.Q * self.C * self.R * self.S

    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def alg_bytes(self, op: str) -> int:
        """Two operands read once plus the result written once."""
        nx = self.N * self.C * self.H * self.W
        ny = self.N * self.K * self.P * self.Q
        nw = self.K * self.C * self.R * self.S
        return (nx + ny + nw) * self.elem_bytes()

    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int          # seed base = 1000 * wid
    problem: Conv2dProblem
    dist: str         # "uniform" (U[-1,1] for x, w, dy) | "he" (x, dy ~ N(0,1); w ~ N(0, 2/CRS)) | "normal"
    description: str


WORKLOADS = {
    "tiny": Workload("tiny", 1, Conv2dProblem(2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1), "uniform",
                     "tiny conv2d fp32: N=2 C=3 H=W=8 K=4 R=S=3 pad 1 stride 1"),
    "resnet3x3": Workload("resnet3x3", 2, Conv2dProblem(32, 64, 56, 56, 64, 3, 3, 1, 1, 1, 1), "he",
                          "ResNet-style 3x3 fp32/TF32: N=32 C=K=64 H=W=56 pad 1 stride 1"),
    "strided": Workload("strided", 3, Conv2dProblem(64, 128, 56, 56, 256, 3, 3, 1, 1, 2, 2), "he",
                        "strided downsample fp32/TF32: N=64 C=128 K=256 H=W=56 3x3 pad 1 stride 2"),
    "pointwise": Workload("pointwise", 41, Conv2dProblem(128, 256, 14, 14, 1024, 1, 1, 0, 0, 1, 1), "he",
                          "1x1 conv fp32/TF32: N=128 C=256 K=1024 H=W=14"),
    "stem7x7": Workload("stem7x7", 42, Conv2dProblem(64, 3, 224, 224, 64, 7, 7, 3, 3, 2, 2), "he",
                        "7x7 stem fp32/TF32: N=64 C=3 K=64 H=W=224 pad 3 stride 2"),
    "deconv": Workload("deconv", 5, Conv2dProblem(32, 256, 32, 32, 512, 4, 4, 1, 1, 2, 2, "bf16"), "normal",
                       "deconvolution bf16: deconv input [32,512,16,16] -> output [32,256,32,32], "
                       "weight [512,256,4,4], 4x4 stride 2 pad 1 (conv view: C=256, K=512, H=W=32)"),
}


def _draw(shape, seed, kind, std=1.0):
    g = torch.Generator().manual_seed(seed)
    if kind == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    return torch.randn(shape, generator=g, dtype=torch.float32) * std


def make_inputs(wl: Workload):
    """(x, w, dy) CPU tensors in the workload's dtype, drawn from seed 1000*wid + {0,1,2}."""
    pb = wl.problem
    base = 1000 * wl.wid
    if wl.dist == "uniform":
        x = _draw(pb.x_shape, base + 0, "uniform")
        w = _draw(pb.w_shape, base + 1, "uniform")
        dy = _draw(pb.y_shape, base + 2, "uniform")
    elif wl.dist == "he":
        x = _draw(pb.x_shape, base + 0, "normal")
        w = _draw(pb.w_shape, base + 1, "normal", math.sqrt(2.0 / (pb.C * pb.R * pb.S)))
        dy = _draw(pb.y_shape, base + 2, "normal")
    else:
        x = _draw(pb.x_shape, base + 0, "normal")
        w = _draw(pb.w_shape, base + 1, "normal")
        dy = _draw(pb.y_shape, base + 2, "normal")
    dt = pb.torch_dtype()
    return x.to(dt), w.to(dt), dy.to(dt)


def random_problem_inputs(pb: Conv2dProblem, seed: int, kind: str = "uniform"):
    """Seeded (x, w, dy) for an arbitrary problem (used by the small parity cases)."""
    dt = pb.torch_dtype()
    return (_draw(pb.x_shape, seed, kind).to(dt),
            _draw(pb.w_shape, seed + 1, kind).to(dt),
            _draw(pb.y_shape, seed + 2, kind).to(dt))
