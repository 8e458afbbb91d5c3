"""Seeded synthetic inputs for the NF4 + LoRA linear layer.

This module only draws random numbers; it holds none of the method's arithmetic.  Both
the CUDA path's tests/benchmark and the CPU oracle take their inputs from here.

Recipe (the shapes and distributions of the QLoRA workloads this library targets):
  * NumPy ``Generator(PCG64(seed))``; seed = 1000 * config + tensor id, tensor ids
    W=1, X=2, A=3, B=4, dY=5, and layer l of a stack adds 10 * l.
  * weights: fp32 N(0, sigma); optionally exactly floor(frac * numel) entries, chosen
    without replacement, replaced by Student-t(3) * 0.1 draws (outliers);
  * activations X, adapters A, B and output gradients dY: fp32 normal draws rounded to
    bf16 (round to nearest even, by torch's dtype conversion) and returned as raw
    uint16 bits.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

TENSOR_IDS = {"W": 1, "X": 2, "A": 3, "B": 4, "dY": 5}


def seed_for(config: int, tensor: str, layer: int = 0) -> int:
    return 1000 * config + TENSOR_IDS[tensor] + 10 * layer


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def weight(shape, seed: int, sigma: float, outlier_frac: float = 0.0) -> np.ndarray:
    """fp32 weights ~ N(0, sigma), with optional Student-t(3) x 0.1 outliers."""
    g = rng(seed)
    w = g.standard_normal(size=shape, dtype=np.float32)
    w *= np.float32(sigma)
    if outlier_frac > 0.0:
        flat = w.reshape(-1)
        k = int(np.floor(outlier_frac * flat.size))
        pos = g.choice(flat.size, size=k, replace=False)
        flat[pos] = (g.standard_t(3, size=k) * 0.1).astype(np.float32)
    return w


def student_t_weight(shape, seed: int, df: float, sigma: float) -> np.ndarray:
    """fp32 heavy-tailed weights: Student-t(df) samples scaled by sigma."""
    g = rng(seed)
    return (g.standard_t(df, size=shape) * sigma).astype(np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_normal(shape, seed: int, sigma: float = 1.0) -> np.ndarray:
    g = rng(seed)
    x = g.standard_normal(size=shape, dtype=np.float32)
    x *= np.float32(sigma)
    return to_bf16_bits(x)


@dataclass
class LinearProblem:
    """One LoRA-wrapped linear layer: W [N,K], X [M,K], A [r,K], B [N,r], dY [M,N]."""
    name: str
    M: int
    N: int
    K: int
    r: int
    alpha: float
    w_sigma: float = 0.02
    outlier_frac: float = 0.0
    config: int = 1
    layer: int = 0
    b_zero: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return self.alpha / self.r

    def W(self) -> np.ndarray:
        return weight((self.N, self.K), seed_for(self.config, "W", self.layer),
                      self.w_sigma, self.outlier_frac)

    def X(self) -> np.ndarray:
        return bf16_normal((self.M, self.K), seed_for(self.config, "X", self.layer), 1.0)

    def A(self) -> np.ndarray:
        return bf16_normal((self.r, self.K), seed_for(self.config, "A", self.layer), 0.01)

    def B(self) -> np.ndarray:
        if self.b_zero:
            return np.zeros((self.N, self.r), np.uint16)
        return bf16_normal((self.N, self.r), seed_for(self.config, "B", self.layer), 0.01)

    def dY(self) -> np.ndarray:
        return bf16_normal((self.M, self.N), seed_for(self.config, "dY", self.layer), 1.0)

    def fwd_flops(self) -> float:
        return 2.0 * self.M * self.N * self.K + 2.0 * self.M * self.r * (self.K + self.N)

    def fwd_bwd_flops(self) -> float:
        return 4.0 * self.M * self.N * self.K + 6.0 * self.M * self.r * (self.K + self.N)


# The five workloads: a small parity case, a 7B attention projection, the 7B MLP
# projections with outliers, a 70B-MLP decode GEMV and a 32-layer 7B stack.
def config1(b_zero: bool = False) -> LinearProblem:
    return LinearProblem("single-linear-256", 16, 256, 256, 8, 16.0, 0.02, config=1,
                         b_zero=b_zero)


def config2() -> LinearProblem:
    return LinearProblem("attn-proj-4096x4096-M4096", 4096, 4096, 4096, 16, 32.0, 0.02,
                         config=2)


def config3() -> list[LinearProblem]:
    return [
        LinearProblem("mlp-gate-11008x4096-M2048", 2048, 11008, 4096, 16, 32.0, 0.02, 0.001,
                      config=3, layer=0),
        LinearProblem("mlp-up-11008x4096-M2048", 2048, 11008, 4096, 16, 32.0, 0.02, 0.001,
                      config=3, layer=1),
        LinearProblem("mlp-down-4096x11008-M2048", 2048, 4096, 11008, 16, 32.0, 0.02, 0.001,
                      config=3, layer=2),
    ]


def config4(M: int) -> LinearProblem:
    assert M in (1, 4, 16)
    return LinearProblem(f"decode-28672x8192-M{M}", M, 28672, 8192, 64, 16.0, 0.015,
                         config=4)


LLAMA7B_PROJ = [("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
                ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008)]


def config5(layer: int, M: int = 512) -> list[LinearProblem]:
    out = []
    for i, (nm, N, K) in enumerate(LLAMA7B_PROJ):
        out.append(LinearProblem(f"llama7b-L{layer}-{nm}", M, N, K, 16, 32.0, 0.02,
                                 config=5, layer=7 * layer + i))
    return out
