"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only draws seeded N(0, 1) tensors
and lists the workload shapes.  It is the one module that both the CUDA path
(tests, bench) and the CPU oracle (tests) use.

Workloads (shapes from "Developing a faster schedule for Longformer's kernel",
posts 3, 4 and 6: hidden 768 = 12 heads x 64, n = 4096, window 512 = 256 on
each side, dilation 0 and 3, sequence lengths up to 512 x 64; 16 global tokens
as in the ONNX Runtime LongformerAttention experiments):

  1  tiny_fp32     b=1  h=2  n=512   hd=64 w=32   w_upper=32  dil=0  fp32
  2  base_fp16     b=1  h=12 n=4096  hd=64 w=256  w_upper=256 dil=0  fp16
  3  dilated_fp16  b=1  h=12 n=4096  hd=64 w=256  w_upper=256 dil=3  fp16
  4  train_bf16    b=12 h=12 n=4096  hd=64 w=256  w_upper=256 dil=0  bf16, 16 global
  5  causal_fp16   b=1  h=12 n=32768 hd=64 w=4096 w_upper=0   dil=0  fp16

Recipe: ``torch.Generator('cpu').manual_seed(1000 + config_id)``, then
``torch.randn`` in fp32 for Q, K, V, dO in that order, each cast to the
workload dtype.  Scale 1/sqrt(64), padding 0.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    config_id: int
    name: str
    b: int
    h: int
    n: int
    head_dim: int
    w: int
    w_upper: int
    dilation: int
    dtype: torch.dtype
    global_idx: tuple = field(default_factory=tuple)
    padding: float = 0.0

    @property
    def BH(self) -> int:
        return self.b * self.h

    @property
    def D(self) -> int:
        return self.w + self.w_upper + 1

    @property
    def scale(self) -> float:
        return 1.0 / (self.head_dim ** 0.5)

    def describe(self) -> dict:
        return {"workload": self.name, "b": self.b, "h": self.h, "n": self.n,
                "head_dim": self.head_dim, "w": self.w, "w_upper": self.w_upper,
                "dilation": self.dilation, "dtype": str(self.dtype).replace("torch.", ""),
                "n_global": len(self.global_idx)}


WORKLOADS = {
    1: Workload(1, "tiny_fp32_n512_w32", 1, 2, 512, 64, 32, 32, 0, torch.float32),
    2: Workload(2, "longformer_base_fp16_n4096_w256_d0", 1, 12, 4096, 64, 256, 256, 0,
                torch.float16),
    3: Workload(3, "longformer_base_fp16_n4096_w256_d3", 1, 12, 4096, 64, 256, 256, 3,
                torch.float16),
    4: Workload(4, "train_bf16_b12_n4096_w256_g16", 12, 12, 4096, 64, 256, 256, 0,
                torch.bfloat16, tuple(range(16))),
    5: Workload(5, "causal_fp16_n32768_w4096", 1, 12, 32768, 64, 4096, 0, 0, torch.float16),
}


def seeded_qkvo(BH: int, n: int, head_dim: int, dtype: torch.dtype, seed: int,
                count: int = 4) -> list[torch.Tensor]:
    """``count`` CPU tensors [BH, n, head_dim] ~ N(0,1) in ``dtype`` (Q, K, V, dO order)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return [torch.randn((BH, n, head_dim), generator=g, dtype=torch.float32).to(dtype)
            for _ in range(count)]


def workload_inputs(wl: Workload, count: int = 4) -> list[torch.Tensor]:
    """The workload's Q, K, V, dO on the CPU, from seed 1000 + config id."""
    return seeded_qkvo(wl.BH, wl.n, wl.head_dim, wl.dtype, 1000 + wl.config_id, count)


def seeded_band(BH: int, n: int, D: int, dtype: torch.dtype, seed: int) -> torch.Tensor:
    """A CPU band tensor [BH, n, D] ~ N(0,1) (input to the band-consuming kernels)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randn((BH, n, D), generator=g, dtype=torch.float32).to(dtype)


def seeded_uniform(shape, dtype: torch.dtype, seed: int, lo: float = 0.0,
                   hi: float = 1.0) -> torch.Tensor:
    """A CPU tensor ~ U(lo, hi) (probability-like band inputs)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo).to(dtype)
