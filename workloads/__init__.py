"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no NVFP4 arithmetic: it only draws bf16 tensors with the
shapes and value distributions of the workloads (Gaussian bodies with a
Bernoulli mask of scaled outliers) and lists those workloads.  Shapes come
from the MaxText Llama 3 8B / Llama 3.1 405B pretraining runs described in the
readjensen.com NVFP4 training-recipe article (sequence 8192, per-device batch
4, so 32768 tokens per GPU); hidden sizes are the public model shapes.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

SEED_X = 0      # activations / A operand
SEED_W = 1      # weights
SEED_DY = 2     # output gradients
RHT_SEED = 7    # shared by both wgrad operands
SR_SEED_BASE = 1000


@dataclass(frozen=True)
class TensorSpec:
    rows: int
    cols: int
    std: float
    outlier_p: float = 0.0
    outlier_factor: float = 1.0
    seed: int = 0


def make_bf16(spec: TensorSpec, device="cpu", base_seed: int = 0) -> torch.Tensor:
    """bf16 [rows, cols] ~ N(0, std^2); a Bernoulli(outlier_p) subset is
    multiplied by outlier_factor.  Deterministic for (spec, device, base_seed)."""
    g = torch.Generator(device=device)
    g.manual_seed(base_seed + spec.seed)
    x = torch.randn(spec.rows, spec.cols, generator=g, device=device, dtype=torch.float32)
    x.mul_(spec.std)
    if spec.outlier_p > 0.0:
        mask = torch.rand(spec.rows, spec.cols, generator=g, device=device) < spec.outlier_p
        x = torch.where(mask, x * spec.outlier_factor, x)
    return x.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """Host uint16 view of a bf16 tensor (numpy), for the oracle."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


@dataclass(frozen=True)
class GemmCase:
    name: str
    a: TensorSpec            # [M, K] before any transpose
    b: TensorSpec            # [N, K] before any transpose
    a_flags: tuple = ()      # quantiser options for A
    b_flags: tuple = ()
    note: str = ""


# Tiny case: A [256,256] ~N(0,1) with 1% x50 outliers, W [256,256] ~N(0,0.02);
# A 1D, W 2D, RNE; C = A W^T.
TINY = GemmCase("tiny_fprop_256",
                TensorSpec(256, 256, 1.0, 0.01, 50.0, SEED_X),
                TensorSpec(256, 256, 0.02, 0.0, 1.0, SEED_W),
                ("1d",), ("2d",))

# Llama 3 8B MLP fprop: X [32768, 4096] ~N(0,1) with 0.1% x30 outliers,
# gate+up W [28672, 4096] ~N(0, 0.02) 2D.
LLAMA3_8B_FPROP = GemmCase("llama3_8b_mlp_fprop",
                           TensorSpec(32768, 4096, 1.0, 0.001, 30.0, SEED_X),
                           TensorSpec(28672, 4096, 0.02, 0.0, 1.0, SEED_W),
                           ("1d",), ("2d",))

# Llama 3 8B MLP backward of one 14336-wide projection:
# dY [32768, 14336] ~N(0, 1e-3), X [32768, 4096] ~N(0,1), W [14336, 4096] ~N(0,0.02).
LLAMA3_8B_DY = TensorSpec(32768, 14336, 1e-3, 0.0, 1.0, SEED_DY)
LLAMA3_8B_X_BWD = TensorSpec(32768, 4096, 1.0, 0.0, 1.0, SEED_X)
LLAMA3_8B_W_BWD = TensorSpec(14336, 4096, 0.02, 0.0, 1.0, SEED_W)

# Llama 3.1 405B MLP fprop: X [8192, 16384] 0.1% x30 outliers, W [106496, 16384] ~N(0,0.01) 2D.
LLAMA31_405B_FPROP = GemmCase("llama31_405b_mlp_fprop",
                              TensorSpec(8192, 16384, 1.0, 0.001, 30.0, SEED_X),
                              TensorSpec(106496, 16384, 0.01, 0.0, 1.0, SEED_W),
                              ("1d",), ("2d",))


def sweep_spec(log2_n: int) -> TensorSpec:
    """Quantise-only sweep: 2^log2_n elements, 4096 rows, ~N(0,1) with 0.1% x100."""
    n = 1 << log2_n
    return TensorSpec(4096, n // 4096, 1.0, 0.001, 100.0, SEED_X)


SWEEP_LOG2 = tuple(range(20, 31))


def sr_seed(k: int) -> int:
    return SR_SEED_BASE + k
