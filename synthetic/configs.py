"""The five synthetic workloads: shapes, dtypes, scales and value distributions.

These describe the DoRA modules the paper write-ups measure on ("Scaling DoRA:
High-Rank Adaptation via Factored Norms and Fused Kernels", section 1.3 for the
8192-square r=512 fp32 memory case, section 3.3 for the 8192x28672 MoE shape,
section 2.1.1 for the magnitude scale g concentrating at mean 1.0, std 0.0015,
and section 2.2 for the small-d_out KV projections of 7B-class models).  No
dataset or trained weights are involved: every tensor is drawn from a seeded
normal distribution by :mod:`synthetic.gen`.

This module holds no DoRA arithmetic; it is shared by the oracle-side tests and
the GPU-side tests/bench only as a description of *what* to generate.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Tuple

BF16 = "bf16"
F32 = "f32"


@dataclass(frozen=True)
class Module:
    """One adapted linear layer: W is [d_out x d_in], A is [r x d_in], B is [d_out x r]."""
    name: str
    d_out: int
    d_in: int


@dataclass(frozen=True)
class Config:
    name: str
    index: int
    dtype: str                 # storage dtype of W, A, B, m, base, lora, out
    modules: Tuple[Module, ...]
    r: int
    s: float
    eps: float
    tokens: int                # compose rows T per module
    std_w: float = 0.02
    std_b: float = 0.01
    std_m_rel: float = 0.0015  # m = ||W||_row * (1 + N(0, std_m_rel))
    std_base: float = 1.0
    std_lora: float = 0.05
    # upstream gradient dL/d out of the compose (training path); the
    # "Scaling DoRA" write-ups give no distribution for it; N(0, 0.01) is
    # chosen here
    std_grad: float = 0.01
    # "norm": compose uses g produced by the norm of the same module;
    # "synthetic": g ~ N(1, g_std) drawn directly (fp32).
    g_mode: str = "norm"
    g_std: float = 0.0015

    def std_a(self, d_in: int) -> float:
        return 1.0 / math.sqrt(d_in)

    @property
    def module(self) -> Module:
        assert len(self.modules) == 1
        return self.modules[0]


def _stack_7b() -> Tuple[Module, ...]:
    h, ffn = 3584, 18944
    mods: List[Module] = []
    for layer in range(28):
        mods += [
            Module(f"L{layer}.q", h, h),
            Module(f"L{layer}.k", 512, h),
            Module(f"L{layer}.v", 512, h),
            Module(f"L{layer}.o", h, h),
            Module(f"L{layer}.gate", ffn, h),
            Module(f"L{layer}.up", ffn, h),
            Module(f"L{layer}.down", h, ffn),
        ]
    return tuple(mods)


CONFIGS: Tuple[Config, ...] = (
    Config("tiny-64x96-r8-f32", 0, F32, (Module("tiny", 64, 96),), r=8, s=2.0,
           eps=1e-6, tokens=32),
    Config("square-8192-r384-bf16", 1, BF16, (Module("square", 8192, 8192),),
           r=384, s=1.0, eps=1e-6, tokens=2048),
    Config("square-8192-r512-f32", 2, F32, (Module("square", 8192, 8192),),
           r=512, s=0.5, eps=1e-6, tokens=4096),
    Config("moe-28672x8192-r384-bf16", 3, BF16, (Module("moe", 28672, 8192),),
           r=384, s=1.0, eps=1e-6, tokens=4096, g_mode="synthetic"),
    Config("stack-7b-196mod-r128-bf16", 4, BF16, _stack_7b(), r=128, s=2.0,
           eps=1e-6, tokens=2048, g_mode="synthetic"),
)

BY_NAME = {c.name: c for c in CONFIGS}


def get(index_or_name) -> Config:
    if isinstance(index_or_name, int):
        return CONFIGS[index_or_name]
    return BY_NAME[index_or_name]


def elem_bytes(dtype: str) -> int:
    return 2 if dtype == BF16 else 4


def norm_flops(d_out: int, d_in: int, r: int) -> int:
    """Algorithmic FLOPs of one factored norm: U = W A^T, G = A A^T, B G, the
    sum of squares of W (one multiply-add per element)."""
    return 2 * d_out * d_in * r + 2 * r * r * d_in + 2 * d_out * r * r + 2 * d_out * d_in


def norm_bytes(d_out: int, d_in: int, r: int, dtype: str) -> int:
    """Algorithmic HBM bytes of one factored norm: read W, A, B, m once; write
    wnorm and g (fp32)."""
    eb = elem_bytes(dtype)
    return eb * (d_out * d_in + r * d_in + d_out * r + d_out) + 8 * d_out


def compose_train_bytes(tokens: int, d_out: int, dtype: str) -> int:
    """Algorithmic bytes of the training forward: read base, lora, g; write
    out and inner."""
    return 4 * tokens * d_out * elem_bytes(dtype) + 4 * d_out


def compose_backward_bytes(tokens: int, d_out: int, dtype: str, dmag: bool = True) -> int:
    """Algorithmic bytes of the backward: read d_out (and inner), g (and
    wnorm); write d_base, d_lora (and dmag)."""
    eb = elem_bytes(dtype)
    n = tokens * d_out
    return (4 * n * eb + 12 * d_out) if dmag else (3 * n * eb + 4 * d_out)


def compose_bytes(tokens: int, d_out: int, dtype: str) -> int:
    """Algorithmic HBM bytes of one compose: read base and lora, write out, read g."""
    eb = elem_bytes(dtype)
    return 3 * tokens * d_out * eb + 4 * d_out
