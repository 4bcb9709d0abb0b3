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
    "LoopShape",
    "LOOP_128",
    "LOOP_SMALL",
    "loop_window",
    "loop_block",
    "loop_undecoded",
    "loop_boosted",
    "loop_planted",
    "loop_offsets",
    "loop_counts",
    "loop_row_cap",
    "make_loop_pools",
    "loop_step_inputs",
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


# --------------------------------------------------------------------------
# Block-wise decoding loop: batch 4, 1024 prompt + 1024 generated positions
# in 32 blocks of 32, 4 partial steps per block (128 steps).
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class LoopShape:
    """Sizes and schedule constants of the block-wise decoding loop.

    The generated positions [prompt, L) form blocks of ``block`` positions,
    decoded one block after the other in ``steps_per_block`` partial steps
    each.  ``n_random`` generated positions per batch row and step are planted
    as salient on top of the current block's undecoded positions; every
    ``refresh``-th step (the first of each block) the selection window is the
    whole sequence, the other steps only the generated rows.  ``boost`` is
    added to the largest logit of the rows whose positions the step should
    commit, ``commit`` of them per step.
    """

    name: str = "bf16_B4_L2048_blocks32_128steps"
    B: int = 4
    L: int = 2048
    H: int = 32
    d: int = 128
    D: int = 4096
    V: int = 126464
    dtype: torch.dtype = torch.bfloat16
    prompt: int = 1024
    block: int = 32
    steps_per_block: int = 4
    commit: int = 8
    n_random: int = 102
    refresh: int = 4
    tau: float = 0.99
    tau_c: float = 0.9
    boost: float = 20.0
    seed: int = 4
    pool_rows: int = 256

    @property
    def T(self) -> int:
        return (self.L - self.prompt) // self.block * self.steps_per_block


LOOP_128 = LoopShape()

# A small loop of the same structure (tests: several blocks in seconds).
LOOP_SMALL = LoopShape(name="bf16_B2_L384_blocks32", B=2, L=384, H=4, d=128, D=256, V=4096,
                       prompt=256, n_random=13, seed=11, pool_rows=64)


def loop_window(shape: LoopShape, s: int) -> int:
    """First position of step s's selection window: 0 (the whole sequence)
    on every ``refresh``-th step, else the prompt length."""
    return 0 if s % shape.refresh == 0 else shape.prompt


def loop_block(shape: LoopShape, s: int):
    """(first position of step s's block, phase j of the step in its block)."""
    k, j = divmod(s, shape.steps_per_block)
    return shape.prompt + k * shape.block, j


def loop_undecoded(shape: LoopShape, s: int):
    """Positions of the current block not yet committed by the schedule at
    step s (``commit`` per earlier step of the block): [lo, hi)."""
    bs, j = loop_block(shape, s)
    return bs + shape.commit * j, bs + shape.block


def loop_boosted(shape: LoopShape, s: int):
    """Positions whose logit rows carry the boost at step s: the first
    ``commit * (j + 1)`` positions of the current block, [lo, hi)."""
    bs, j = loop_block(shape, s)
    return bs, bs + shape.commit * (j + 1)


def loop_planted(shape: LoopShape, s: int):
    """Sorted absolute positions planted as salient at step s, per batch row:
    the block's undecoded positions and ``n_random`` generated positions
    drawn uniformly without replacement (a generator seeded per step)."""
    g = torch.Generator().manual_seed(shape.seed * 1000003 + 7919 * s)
    lo, hi = loop_undecoded(shape, s)
    block_part = torch.arange(lo, hi)
    out = []
    for _ in range(shape.B):
        rnd = torch.randperm(shape.L - shape.prompt, generator=g)[:shape.n_random] + shape.prompt
        out.append(torch.unique(torch.cat([block_part, rnd])))  # sorted
    return out


def loop_offsets(shape: LoopShape, s: int):
    """Per-step starting rows in the fresh-row and logit pools, [B] each."""
    g = torch.Generator().manual_seed(shape.seed * 1000003 + 7919 * s + 1)
    return (torch.randint(0, shape.pool_rows, (shape.B,), generator=g),
            torch.randint(0, shape.pool_rows, (shape.B,), generator=g))


def loop_counts(shape: LoopShape):
    """Planted counts [T, B] of every step (host schedule, no tensors drawn
    beyond the position sets)."""
    return torch.tensor([[len(p) for p in loop_planted(shape, s)] for s in range(shape.T)],
                        dtype=torch.int64)


def loop_row_cap(shape: LoopShape) -> int:
    """Logit rows per batch row every step's buffer holds: the largest planted
    count of the schedule."""
    return int(loop_counts(shape).max())


def make_loop_pools(shape: LoopShape) -> dict:
    """Everything the loop's steps are assembled from, as CPU tensors.

    ``prev`` [B, L, D] ~ N(0, 1) is the cached hidden state of every
    position; ``hot`` = prev + N(0, 0.5) and ``cold`` = prev + N(0, 1e-3)
    are a position's current hidden state when planted salient or not (the
    sums taken in float64, then cast); ``k_cache``/``v_cache`` [B, L, H, d]
    the cache before the first step; ``q_pool``/``k_pool``/``v_pool``
    [B, pool_rows, H, d] fresh query/key/value rows, all N(0, 1);
    ``logit_pool`` [B, pool_rows, V] ~ N(0, 2) and ``boost_pool``, the same
    rows with ``boost`` added to each row's largest logit (its lowest index
    on a tie), in float64 and then cast.
    """
    g = torch.Generator().manual_seed(shape.seed)
    B, L, H, d, D, V, R = shape.B, shape.L, shape.H, shape.d, shape.D, shape.V, shape.pool_rows
    dt = shape.dtype
    prev64 = torch.randn((B, L, D), generator=g, dtype=torch.float64)
    hot = (prev64 + torch.randn((B, L, D), generator=g, dtype=torch.float64) * 0.5).to(dt)
    cold = (prev64 + torch.randn((B, L, D), generator=g, dtype=torch.float64) * 1e-3).to(dt)
    prev = prev64.to(dt)
    del prev64
    pools = dict(prev=prev, hot=hot, cold=cold,
                 k_cache=normal(g, (B, L, H, d), 1.0, dt), v_cache=normal(g, (B, L, H, d), 1.0, dt),
                 q_pool=normal(g, (B, R, H, d), 1.0, dt), k_pool=normal(g, (B, R, H, d), 1.0, dt),
                 v_pool=normal(g, (B, R, H, d), 1.0, dt))
    logit_pool = normal(g, (B, R, V), 2.0, dt)
    boost_pool = logit_pool.clone()
    top = torch.argmax(logit_pool.float(), dim=-1)  # first index of the maximum
    rows = torch.arange(R)
    for b in range(B):
        v = logit_pool[b, rows, top[b]].double() + shape.boost
        boost_pool[b, rows, top[b]] = v.to(dt)
    pools["logit_pool"] = logit_pool
    pools["boost_pool"] = boost_pool
    return pools


def loop_step_inputs(shape: LoopShape, pools: dict, s: int, row_cap: int,
                     device=None) -> dict:
    """Inputs of step s, assembled on ``device`` from pools that live there.

    Only selection and indexing: the same pools give the same bits on the
    CPU and on a GPU.  ``cur`` [B, L, D]: ``hot`` at the planted positions,
    ``cold`` elsewhere; ``k_new``/``v_new`` [B, Lw, H, d] (Lw = the
    window's length, the layout of the compacted indices) and ``q``
    [B, row_cap, H, d]: row i < count[b] is pool row (offset + i) mod
    pool_rows, the rest zero; ``logits`` [B, row_cap, V]: row r < count[b] is
    logit-pool row (offset + r) mod pool_rows, from ``boost_pool`` when the
    r-th planted position lies in the boosted range, the rest zero.
    Also returns ``win_start``, ``planted`` (CPU) and ``counts`` (list).
    """
    dev = pools["prev"].device if device is None else device
    planted = loop_planted(shape, s)
    off_kv, off_l = loop_offsets(shape, s)
    w = loop_window(shape, s)
    Lw = shape.L - w
    B, L, H, d, V, R = shape.B, shape.L, shape.H, shape.d, shape.V, shape.pool_rows
    mask = torch.zeros((B, L), dtype=torch.bool)
    for b in range(B):
        mask[b, planted[b]] = True
    cur = torch.where(mask.to(dev)[:, :, None], pools["hot"], pools["cold"])
    q = torch.zeros((B, row_cap, H, d), dtype=shape.dtype, device=dev)
    k_new = torch.zeros((B, Lw, H, d), dtype=shape.dtype, device=dev)
    v_new = torch.zeros_like(k_new)
    logits = torch.zeros((B, row_cap, V), dtype=shape.dtype, device=dev)
    blo, bhi = loop_boosted(shape, s)
    for b in range(B):
        n = len(planted[b])
        if n > row_cap:
            raise ValueError(f"step {s}: {n} planted rows exceed the logit buffer's {row_cap}")
        rows = ((int(off_kv[b]) + torch.arange(n)) % R).to(dev)
        q[b, :n] = pools["q_pool"][b].index_select(0, rows)
        k_new[b, :n] = pools["k_pool"][b].index_select(0, rows)
        v_new[b, :n] = pools["v_pool"][b].index_select(0, rows)
        lrows = ((int(off_l[b]) + torch.arange(n)) % R).to(dev)
        boosted = ((planted[b] >= blo) & (planted[b] < bhi)).to(dev)
        plain = pools["logit_pool"][b].index_select(0, lrows)
        hot_rows = pools["boost_pool"][b].index_select(0, lrows)
        logits[b, :n] = torch.where(boosted[:, None], hot_rows, plain)
    return dict(cur=cur, q=q, k_new=k_new, v_new=v_new, logits=logits, win_start=w,
                planted=planted, counts=[len(p) for p in planted])
