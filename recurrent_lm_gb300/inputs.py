"""Seeded synthetic inputs for causal Taylor linear attention workloads.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so that the GPU path and the CPU oracle can both be fed
from it without sharing any computation.

The workloads stand in for the pages' timing runs (which used random inputs):
H = 16 heads with d' = 16 follow the BASED model configuration table, d_v = 64
is hidden 1024 / 16 heads, batch 16 and N up to 32768 follow the prefill
latency table of the "Just read twice" page, and decode batch 128 follows the
BASED decode throughput run.  Values are N(0, 1) (config 2: scaled by
1/sqrt(2)), drawn in fp32 with a CPU torch.Generator and cast to the
activation dtype with round-to-nearest-even.  Draw order: q, k, v, then the
prefix set k_e, v_e.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

D_FEAT = 16   # d'
D_V = 64      # d_v


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int            # causal tokens (decode: 1 per step)
    dtype: torch.dtype
    scale: float = 1.0
    M: int = 0        # prefix length (JRT-RNN)
    s0_tokens: int = 0  # length of the seeded sequence whose final state seeds s0
    steps: int = 0    # decode steps
    seed: int = 0


WORKLOADS = {
    1: Workload("causal-fp32-B1-H2-N256", 1, 2, 256, torch.float32, seed=1001),
    2: Workload("based-prefill-bf16-B8-H16-N2048", 8, 16, 2048, torch.bfloat16,
                scale=1.0 / math.sqrt(2.0), seed=1002),
    3: Workload("long-prefill-bf16-B16-H16-N32768-s0from4096", 16, 16, 32768,
                torch.bfloat16, s0_tokens=4096, seed=1003),
    4: Workload("jrt-prefix-bf16-B16-H16-N32768-M16384", 16, 16, 32768,
                torch.bfloat16, M=16384, seed=1004),
    5: Workload("decode-bf16-B128-H16-512steps-from2048", 128, 16, 1,
                torch.bfloat16, s0_tokens=2048, steps=512, seed=1005),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn(shape, g: torch.Generator, dtype: torch.dtype, scale: float = 1.0):
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(dtype)


def qkv(B: int, H: int, N: int, seed: int, dtype=torch.bfloat16, scale: float = 1.0,
        dk: int = D_FEAT, dv: int = D_V, M: int = 0):
    """(q, k, v, ke, ve) on the CPU; ke/ve are None when M == 0."""
    g = _gen(seed)
    q = randn((B, H, N, dk), g, dtype, scale)
    k = randn((B, H, N, dk), g, dtype, scale)
    v = randn((B, H, N, dv), g, dtype, scale)
    ke = ve = None
    if M > 0:
        ke = randn((B, H, M, dk), g, dtype, scale)
        ve = randn((B, H, M, dv), g, dtype, scale)
    return q, k, v, ke, ve


def workload_inputs(cfg: int, N: int | None = None, B: int | None = None):
    """Main inputs of a workload (optionally with B or N overridden)."""
    w = WORKLOADS[cfg]
    return qkv(B or w.B, w.H, N or w.N, w.seed, w.dtype, w.scale, M=w.M)


def s0_sequence(cfg: int, B: int | None = None):
    """The separately seeded sequence whose final state seeds s0 (configs 3, 5)."""
    w = WORKLOADS[cfg]
    q, k, v, _, _ = qkv(B or w.B, w.H, w.s0_tokens, 2000 + cfg, w.dtype, w.scale)
    return q, k, v


def decode_step_inputs(cfg: int, step: int, B: int | None = None):
    """Fresh N(0,1) q, k [B,H,d'] and v [B,H,d_v] for decode step ``step``."""
    w = WORKLOADS[cfg]
    g = _gen(5000 + step)
    B = B or w.B
    q = randn((B, w.H, D_FEAT), g, w.dtype)
    k = randn((B, w.H, D_FEAT), g, w.dtype)
    v = randn((B, w.H, D_V), g, w.dtype)
    return q, k, v


def random_state(B: int, H: int, seed: int, D: int = 1 + D_FEAT + D_FEAT * D_FEAT,
                 dv: int = D_V, tokens: float = 64.0):
    """An arbitrary fp32 (s0, z0) for edge-case tests: s0 ~ N(0, tokens), and a
    z0 whose constant entry is ``tokens`` (as after that many tokens) and whose
    other entries are small, so the denominator stays positive."""
    g = _gen(seed)
    s0 = randn((B, H, D, dv), g, torch.float32, math.sqrt(tokens))
    z0 = randn((B, H, D), g, torch.float32, 0.05)
    z0[..., 0] = tokens
    return s0, z0
