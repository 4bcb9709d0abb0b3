"""Seeded synthetic inputs for one partial denoising step.

This module only draws random numbers, casts them and lays the buffers out.  It
holds none of the method's arithmetic, so both the float64 oracle and the CUDA
path can take their inputs from it without sharing any computation.

The shapes stand in for the workloads the pages measure on (LLaDA-8B /
Dream-7B decoding GSM8K-style prompts: 32 heads x 128, hidden 4096, vocabulary
126464).  Neither the models nor the datasets exist here; every tensor is drawn
from a seeded ``torch.Generator`` in float64 and then cast to the step's dtype,
so the oracle sees exactly the bits the GPU sees (the cast to float64 of a
bfloat16 or float32 value is exact).

Recipe (std, not variance, in every N(0, s)):

* hidden states ``prev`` ~ N(0, 1); ``cur = prev + N(0, 0.5)`` on the planted
  salient positions and ``prev + N(0, 1e-3)`` elsewhere;
* K/V cache, fresh K/V rows and the active query rows ~ N(0, 1);
* vocabulary logits ~ N(0, 2);
* salient positions: uniform without replacement inside the selection window
  (``random``) or runs of 32 positions in randomly chosen, non-overlapping,
  32-aligned slots (``cluster``, the contiguous-cluster pattern).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = [
    "StepShape",
    "TINY_F32",
    "STEP_1K",
    "BATCH8_2K",
    "LONG_4K",
    "LOOP_B4_2K",
    "SHAPES",
    "make_step",
    "plant_positions",
    "normal",
]


@dataclasses.dataclass(frozen=True)
class StepShape:
    """Sizes of one partial step.

    B batch, L sequence length, H heads, d head dim, D hidden size, V vocabulary
    size, ``win_start`` the first position of the selection window (the prompt
    length when only the generated rows are scored), ``n_salient`` the planted
    salient positions per batch row, ``tau`` the cosine threshold.
    """

    name: str
    B: int
    L: int
    H: int
    d: int
    D: int
    V: int
    dtype: torch.dtype
    win_start: int
    n_salient: int
    tau: float
    seed: int
    logit_rows: int  # logit rows per batch row (over the window)

    @property
    def Lw(self) -> int:
        return self.L - self.win_start


# Tiny float32 step: 16 salient of 64 positions, 2 heads of 32, vocabulary 256.
TINY_F32 = StepShape("tiny_f32_L64", B=1, L=64, H=2, d=32, D=64, V=256,
                     dtype=torch.float32, win_start=0, n_salient=16, tau=0.99,
                     seed=0, logit_rows=64)

# bf16 step: 512 prompt + 512 generated positions, ~10% of L salient (drawn from
# the generated rows), logits over the generated rows.
STEP_1K = StepShape("bf16_L1024_h32x128_V126464", B=1, L=1024, H=32, d=128,
                    D=4096, V=126464, dtype=torch.bfloat16, win_start=512,
                    n_salient=102, tau=0.99, seed=1, logit_rows=512)

# bf16 batch 8 x 2048; the active fraction is swept, so n_salient is set per call.
BATCH8_2K = StepShape("bf16_B8_L2048_h32x128", B=8, L=2048, H=32, d=128, D=4096,
                      V=126464, dtype=torch.bfloat16, win_start=0, n_salient=205,
                      tau=0.99, seed=2, logit_rows=0)

# bf16 long context: batch 1, L=4096 (64-step lock schedule).
LONG_4K = StepShape("bf16_L4096_h32x128_V126464", B=1, L=4096, H=32, d=128,
                    D=4096, V=126464, dtype=torch.bfloat16, win_start=0,
                    n_salient=4096, tau=2.0, seed=3, logit_rows=4096)

# bf16 loop: batch 4, 1024 prompt + 1024 generated positions.
LOOP_B4_2K = StepShape("bf16_B4_L2048_h32x128_V126464", B=4, L=2048, H=32, d=128,
                       D=4096, V=126464, dtype=torch.bfloat16, win_start=1024,
                       n_salient=102, tau=0.99, seed=4, logit_rows=1024)

SHAPES = {s.name: s for s in (TINY_F32, STEP_1K, BATCH8_2K, LONG_4K, LOOP_B4_2K)}


def normal(g: torch.Generator, shape, std: float, dtype: torch.dtype) -> torch.Tensor:
    """N(0, std) drawn in float64 from ``g`` and cast to ``dtype``."""
    return (torch.randn(shape, generator=g, dtype=torch.float64) * std).to(dtype)


def plant_positions(g: torch.Generator, Lw: int, n: int, pattern: str) -> torch.Tensor:
    """Sorted window-relative positions of ``n`` planted salient rows."""
    if n <= 0:
        return torch.zeros(0, dtype=torch.int64)
    n = min(n, Lw)
    if pattern == "random":
        pos = torch.randperm(Lw, generator=g)[:n]
    elif pattern == "cluster":
        run = 32
        slots = Lw // run
        n_runs = math.ceil(n / run)
        if n_runs > slots:
            raise ValueError("window too short for the requested clusters")
        chosen = torch.randperm(slots, generator=g)[:n_runs]
        parts = [torch.arange(int(s) * run, int(s) * run + run) for s in chosen]
        pos = torch.cat(parts)[:n]
    else:
        raise ValueError(f"unknown pattern {pattern!r}")
    return torch.sort(pos).values


def make_step(shape: StepShape, *, n_salient: Optional[int] = None,
              pattern: str = "random", seed: Optional[int] = None,
              with_logits: bool = True, m_max: Optional[int] = None) -> dict:
    """All inputs of one partial step, as CPU tensors.

    Returned keys: ``cur``/``prev`` [B, L, D]; ``planted`` list of sorted
    absolute positions per batch row; ``k_cache``/``v_cache`` [B, L, H, d];
    ``k_new``/``v_new``/``q`` [B, M_max, H, d]; ``logits`` [B, R, V] (R =
    ``shape.logit_rows``) when ``with_logits``; scalars ``tau``, ``win_start``.
    """
    g = torch.Generator().manual_seed(shape.seed if seed is None else seed)
    B, L, H, d, D = shape.B, shape.L, shape.H, shape.d, shape.D
    dt = shape.dtype
    n = shape.n_salient if n_salient is None else n_salient
    Mmax = shape.Lw if m_max is None else m_max

    prev64 = torch.randn((B, L, D), generator=g, dtype=torch.float64)
    noise = torch.randn((B, L, D), generator=g, dtype=torch.float64) * 1e-3
    planted = []
    for b in range(B):
        rel = plant_positions(g, shape.Lw, n, pattern)
        absolute = rel + shape.win_start
        big = torch.randn((len(absolute), D), generator=g, dtype=torch.float64) * 0.5
        noise[b, absolute] = big
        planted.append(absolute)
    cur = (prev64 + noise).to(dt)
    prev = prev64.to(dt)
    del prev64, noise

    out = dict(
        cur=cur, prev=prev, planted=planted,
        k_cache=normal(g, (B, L, H, d), 1.0, dt),
        v_cache=normal(g, (B, L, H, d), 1.0, dt),
        k_new=normal(g, (B, Mmax, H, d), 1.0, dt),
        v_new=normal(g, (B, Mmax, H, d), 1.0, dt),
        q=normal(g, (B, Mmax, H, d), 1.0, dt),
        tau=shape.tau, win_start=shape.win_start, m_max=Mmax,
    )
    if with_logits and shape.logit_rows > 0:
        out["logits"] = normal(g, (B, shape.logit_rows, shape.V), 2.0, dt)
    return out
