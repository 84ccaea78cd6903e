"""Seeded synthetic inputs for the W4A16 workloads.

This module only draws random numbers and casts them to bf16; it holds none
of the quantization or GEMM arithmetic, so the CUDA library and the CPU
oracle can both be fed from it without sharing any of the method.

Recipe (one reading of the workload descriptions, applied everywhere):

* ``rng = numpy.random.default_rng(seed)``; the weight W[N, K] is drawn
  first, then the activations A[M, K], then (only when asked) a bias[N].
* W: float32 N(0, 1) * 0.02, or Student-t with 4 degrees of freedom * 0.02
  (heavy tails, so single large elements set their group's scale); cast to
  bf16 with round-to-nearest-even.
* A: float32 N(0, 1) cast to bf16.  Bias: float32 N(0, 1) * 0.5 cast to bf16.

The named workloads mirror the shapes of the pi0.5 action expert and
language-model prefix described in "Kernel dispatch and Humming quantization
in PhyAI", section "Humming makes the separation useful" (attention and MLP
projections quantized to INT4, group 128).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Case:
    name: str
    M: int
    N: int
    K: int
    seed: int
    wdist: str = "normal"   # "normal" or "t4"
    bias: bool = False


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """float32 numpy -> bf16 CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def to_f16(x: np.ndarray) -> torch.Tensor:
    """float32 numpy -> fp16 CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float16)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a bf16/fp16 CPU tensor as a uint16 numpy array."""
    if t.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("expected a 16-bit float tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def draw_weight(rng: np.random.Generator, N: int, K: int, wdist: str) -> np.ndarray:
    if wdist == "normal":
        w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    elif wdist == "t4":
        w = (rng.standard_t(4, size=(N, K)) * 0.02).astype(np.float32)
    else:
        raise ValueError(f"unknown weight distribution {wdist!r}")
    return w


def draw(case: Case, act: str = "bf16"):
    """Return ``(W bf16 [N,K], A [M,K], bias [N] or None)`` on CPU; A and the
    bias in the activation type ``act`` ("bf16" or "f16"), from the same
    float32 draws."""
    rng = np.random.default_rng(case.seed)
    cast = to_bf16 if act == "bf16" else to_f16
    w = to_bf16(draw_weight(rng, case.N, case.K, case.wdist))
    a = cast(rng.standard_normal((case.M, case.K), dtype=np.float32))
    b = None
    if case.bias:
        b = cast(rng.standard_normal(case.N, dtype=np.float32) * np.float32(0.5))
    return w, a, b


def draw_weight_only(seed: int, N: int, K: int, wdist: str = "normal") -> torch.Tensor:
    """The weight of ``draw`` alone (same stream position: drawn first)."""
    rng = np.random.default_rng(seed)
    return to_bf16(draw_weight(rng, N, K, wdist))


# The five workloads.  Seeds: the action-expert shapes take seeds 1..4 in the
# listed order; every other workload takes seed 0.
TINY = [Case("tiny_m16_n256_k512", 16, 256, 512, 0)]

EXPERT_M50 = [
    Case("expert_qkv_m50_n2048_k1024", 50, 2048, 1024, 1),
    Case("expert_o_m50_n1024_k1024", 50, 1024, 1024, 2),
    Case("expert_gate_up_m50_n8192_k1024", 50, 8192, 1024, 3),
    Case("expert_down_m50_n1024_k4096", 50, 1024, 4096, 4),
]

PREFIX_M816 = [
    Case("prefix_qkv_m816_n2560_k2048", 816, 2560, 2048, 0, "t4"),
    Case("prefix_o_m816_n2048_k2048", 816, 2048, 2048, 0, "t4"),
    Case("prefix_gate_up_m816_n32768_k2048", 816, 32768, 2048, 0, "t4"),
    Case("prefix_down_m816_n2048_k16384", 816, 2048, 16384, 0, "t4"),
]

SWEEP = [
    Case(f"sweep_m{m}_n{n}_k{k}", m, n, k, 0)
    for (n, k) in ((16384, 2048), (2048, 16384), (8192, 8192))
    for m in (1, 4, 16, 64)
]

LARGE = [Case("large_m8192_n8192_k8192", 8192, 8192, 8192, 0)]

WORKLOADS = {
    "tiny": TINY,
    "expert_m50": EXPERT_M50,
    "prefix_m816": PREFIX_M816,
    "sweep": SWEEP,
    "large": LARGE,
}
