"""Seeded synthetic inputs shared by the tests, the smoke check and the
benchmark. Random numbers only: this module holds none of the method's
arithmetic. Both the CUDA path and the CPU oracle are given the same fp16 (or
bf16) bit patterns generated here.

Recipe: ``torch.Generator(device).manual_seed(seed)``, draw fp32, scale,
round once to fp16 or bf16 (round to nearest even). Seeds are
``config_index * 1000 + tensor_index`` (A = 1, B = 2, bias = 3, dY = 4).
Large tensors are drawn on the GPU (the CPU generator would take minutes);
small ones on the CPU. The workloads stand in for the pages' shapes: the
nvmath-python example (m, n, k = 1024, 512, 2048 with uniform [0,1) data),
the LLaMA FFN projections of the ops-nn article (hidden 4096), a LLaMA-7B
MLP (11008 x 4096) and the large 65536 x 16384 x 8192 product.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

# Largest value below 1 of each 16-bit type: keeps uniform [0,1) draws below 1
# after rounding.
_BELOW_ONE = {torch.float16: 0.99951171875, torch.bfloat16: 0.99609375}

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}


def f16_tensor(shape, seed: int, dist: str = "normal", std: float = 1.0, device="cpu",
               dtype: torch.dtype = torch.float16) -> torch.Tensor:
    """16-bit tensor of `shape` (fp16, or bf16 with dtype=torch.bfloat16):
    dist "normal" -> N(0, std^2); "uniform01" -> U[0,1); "int" -> integers in
    [-std, std]. The same seed gives the same fp32 draws for either type."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    if dist == "uniform01":
        x = torch.rand(shape, generator=g, device=dev, dtype=torch.float32)
        return x.to(dtype).clamp_(max=_BELOW_ONE[dtype])
    if dist == "normal":
        x = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(dtype)
    if dist == "int":  # integers in [-std, std] (exact-arithmetic cases)
        hi = int(std)
        x = torch.randint(-hi, hi + 1, shape, generator=g, device=dev, dtype=torch.int32)
        return x.to(dtype)
    raise ValueError(dist)


def sample_rows(n_rows: int, count: int = 256, seed: int = 0xB0A7) -> np.ndarray:
    """`count` distinct row indices of [0, n_rows), sorted (all rows if fewer)."""
    if n_rows <= count:
        return np.arange(n_rows)
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(n_rows, size=count, replace=False))


@dataclass
class Workload:
    """One canonical problem D[M,N] = act(A.B + bias) with its storage."""
    name: str
    M: int
    N: int
    K: int
    epilogue: str
    a_major: str  # "k" | "m"
    b_major: str  # "k" | "n"
    d_layout: str  # "row" | "col"
    a_dist: tuple = ("normal", 1.0)
    b_dist: tuple = ("normal", 1.0)
    bias_dist: tuple = ("normal", 1.0)
    index: int = 0
    extra: dict = field(default_factory=dict)
    dtype: str = "f16"  # element type of A, B, bias and D: "f16" | "bf16"

    def a_shape(self):
        return (self.M, self.K) if self.a_major == "k" else (self.K, self.M)

    def b_shape(self):
        return (self.N, self.K) if self.b_major == "k" else (self.K, self.N)

    def d_shape(self):
        return (self.M, self.N) if self.d_layout == "row" else (self.N, self.M)

    def make(self, device="cpu"):
        """(A, B, bias) tensors of the workload's element type in storage layout."""
        i = self.index * 1000
        t = TORCH_DTYPE[self.dtype]
        A = f16_tensor(self.a_shape(), i + 1, self.a_dist[0], self.a_dist[1], device, t)
        B = f16_tensor(self.b_shape(), i + 2, self.b_dist[0], self.b_dist[1], device, t)
        bias = f16_tensor((self.M,), i + 3, self.bias_dist[0], self.bias_dist[1], device, t)
        return A, B, bias

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def algorithmic_bytes(self) -> int:
        """Operands read once, D written once, bias read, mask written."""
        b = 2 * (self.M * self.K + self.K * self.N + self.M * self.N) + 2 * self.M
        if self.epilogue == "relu_aux_bias":
            rows, cols = self.d_shape()
            b += rows * ((cols + 127) // 128) * 16
        return b


def pages_workloads():
    """The five workload families (sizes fixed by the pages' examples)."""
    w = {}
    w["c1"] = Workload("c1 PR1 256x128x512 BIAS", 256, 128, 512, "bias", "k", "n", "row",
                       ("uniform01", 1), ("uniform01", 1), ("uniform01", 1), index=0)
    for j, e in enumerate(("bias", "relu_bias", "gelu_bias")):
        w[f"c2_{e}"] = Workload(f"c2 linear 1024x512x2048 {e.upper()}", 1024, 512, 2048, e, "k", "n",
                                "row", ("normal", 1 / math.sqrt(2048)), ("normal", 1 / math.sqrt(2048)),
                                ("normal", 1.0), index=1)
    for T in (1, 512, 2048):
        w[f"c3_T{T}"] = Workload(f"c3 FFN up GELU_BIAS T={T} 4096x{T}x4096", 4096, T, 4096, "gelu_bias",
                                 "k", "k", "col", ("normal", 1 / 64), ("normal", 1.0),
                                 ("normal", math.sqrt(0.02)), index=2)
    w["c4_fwd"] = Workload("c4 MLP fwd RELU_AUX_BIAS 11008x8192x4096", 11008, 8192, 4096,
                           "relu_aux_bias", "k", "k", "col", ("normal", 1 / 64), ("normal", 1.0),
                           ("normal", math.sqrt(0.02)), index=3)
    w["c4_dw"] = Workload("c4 MLP dW 11008x4096x8192 NONE", 11008, 4096, 8192, "none", "m", "n",
                          "row", index=3)
    w["c5"] = Workload("c5 large RELU_AUX_BIAS 65536x8192x16384", 65536, 8192, 16384, "relu_aux_bias",
                       "k", "n", "row", ("normal", 1 / 128), ("normal", 1 / 128), ("normal", 1.0),
                       index=4)
    return w
