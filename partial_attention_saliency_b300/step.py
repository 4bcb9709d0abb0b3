"""One partial denoising step composed from the five library calls.

The order follows the pages: select the salient rows of the window (DyLLM),
write their fresh K/V into the cache (SureLock), attend from them over the
whole cache with per-key column sums (DyLLM, Attn-Sampler), score the window's
logit rows (SlowFast, SureLock, LSP) and find the committable prefix (LSP).
Model work between the calls (Q/K/V projections, FFN, LM head of the active
rows) is outside this library: its results arrive as inputs.

All buffers are allocated once, through torch, in ``__init__``; ``run`` only
launches kernels on the current stream and reads nothing back, so it can be
captured in a CUDA graph.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib


class PartialStep:
    """Device buffers and launches of one partial step.

    B batch, L sequence, H x d heads, D hidden, V vocabulary; the selection
    window is positions [win_start, L) (M_max = L - win_start active rows at
    most); ``logit_rows`` logit rows per batch row cover the window's first
    positions.
    """

    def __init__(self, B: int, L: int, H: int, d: int, D: int, V: int, dtype: torch.dtype,
                 win_start: int, logit_rows: int, tau: float, tau_c: float = 0.9,
                 min_commit: bool = True, colsum: bool = True,
                 device: Optional[torch.device] = None):
        dev = torch.device("cuda") if device is None else device
        self.B, self.L, self.H, self.d, self.D, self.V = B, L, H, d, D, V
        self.dtype, self.win_start, self.logit_rows = dtype, win_start, logit_rows
        self.Lw = L - win_start
        self.M_max = self.Lw
        self.tau, self.tau_c, self.min_commit, self.want_colsum = tau, tau_c, min_commit, colsum
        f32, i32 = torch.float32, torch.int32
        self.cos = torch.empty((B, self.Lw), dtype=f32, device=dev)
        self.idx = torch.empty((B, self.Lw), dtype=i32, device=dev)
        self.count = torch.empty((B,), dtype=i32, device=dev)
        self.o = torch.empty((B, self.M_max, H, d), dtype=dtype, device=dev)
        self.lse = torch.empty((B, H, self.M_max), dtype=f32, device=dev)
        self.colsum = torch.empty((B, H, L), dtype=f32, device=dev) if colsum else None
        self.argmax = torch.zeros((B, L), dtype=i32, device=dev)
        self.margin = torch.zeros((B, L), dtype=f32, device=dev)
        self.length = torch.empty((B,), dtype=i32, device=dev)
        self.dev_status = torch.zeros((1,), dtype=i32, device=dev)
        conf_ws = _lib.dllm_confidence_workspace_bytes(B, max(logit_rows, 1), V, dtype)
        self.conf_ws = torch.empty((max(conf_ws, 16),), dtype=torch.uint8, device=dev)
        attn_ws = _lib.dllm_attention_workspace_bytes(B, L, H, d, self.M_max, dtype)
        self.attn_ws = torch.empty((max(attn_ws, 16),), dtype=torch.uint8, device=dev)

    def run(self, cur, prev, k_cache, v_cache, k_new, v_new, q, logits, score, start,
            stream=None):
        """Launch the step.  ``score`` [B, L] f32 and ``start`` [B] i32 are
        updated in place (confidence over the window rows, then start is not
        advanced: ``self.length`` holds the committable prefix length)."""
        w = self.win_start
        _lib.dllm_saliency_select(cur[:, w:], prev[:, w:], self.tau, idx_base=w,
                                  cos_out=self.cos, idx_out=self.idx, count_out=self.count,
                                  dev_status=self.dev_status, stream=stream)
        _lib.dllm_kv_scatter(k_cache, v_cache, k_new, v_new, self.idx, self.count,
                             dev_status=self.dev_status, stream=stream)
        _lib.dllm_partial_attention(q, k_cache, v_cache, self.count, o_out=self.o,
                                    lse_out=self.lse, colsum_out=self.colsum,
                                    with_colsum=self.want_colsum, ws=self.attn_ws,
                                    dev_status=self.dev_status, stream=stream)
        if logits is not None and self.logit_rows > 0:
            _lib.dllm_confidence(logits, out_cols=self.L, conf_out=score[:, w:],
                                 argmax_out=self.argmax[:, w:], margin_out=self.margin[:, w:],
                                 ws=self.conf_ws, dev_status=self.dev_status, stream=stream)
        _lib.dllm_stable_prefix(score, start, self.tau_c, min_commit=self.min_commit,
                                advance_start=False, len_out=self.length,
                                dev_status=self.dev_status, stream=stream)
        return self
