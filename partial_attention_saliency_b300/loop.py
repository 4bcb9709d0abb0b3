"""Block-wise decoding loop built from the library's calls, one partial step per call.

Per step, in the order the pages give: select the salient rows of the window
(DyLLM; the window is the generated rows on most steps and the whole sequence
every few steps, DyLLM's adaptive input), write their fresh K/V into the
cache (SureLock), attend from them over the whole cache and take the
per-key column sums (DyLLM, Attn-Sampler), score their logit rows (SlowFast,
SureLock, LSP) into the per-position score, and commit the longest stable
prefix from ``start``, advancing it (LSP, at least one token per step).

State carried from step to step stays on the device: the K/V cache, the
per-position score (the confidence of each position's latest prediction)
and ``start``.  Nothing is read back to the host, so any run of steps can be
captured in one CUDA graph.  Model work between the calls (projections, FFN,
LM head of the active rows) is outside the library: its results arrive as
each step's inputs.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import _lib


class BlockDecodeLoop:
    """Device state and buffers of the loop, allocated once.

    B batch rows of L positions, the first ``prompt`` of them committed from
    the start; H x d heads; V vocabulary; ``row_cap`` the most active rows a
    step can have per batch row (the rows of a step's query and logit
    buffers, and of the attention outputs); ``tau`` the cosine threshold,
    ``tau_c`` the confidence a position needs to be committed.

    The attention gets no workspace when B * H already covers half the SMs:
    it then never splits the key range, so no merge launch follows it.

    The column sums feed nothing later in the step, so they run on a second
    stream, concurrently with the confidence and the prefix commit; the step
    joins the two streams before it returns (a fork and a join in a captured
    graph).
    """

    def __init__(self, B: int, L: int, H: int, d: int, V: int, dtype: torch.dtype,
                 prompt: int, row_cap: int, tau: float, tau_c: float,
                 device: Optional[torch.device] = None):
        dev = torch.device("cuda") if device is None else device
        self.B, self.L, self.H, self.d, self.V = B, L, H, d, V
        self.dtype, self.prompt, self.row_cap = dtype, prompt, row_cap
        self.tau, self.tau_c = tau, tau_c
        f32, i32 = torch.float32, torch.int32
        self.k_cache = torch.zeros((B, L, H, d), dtype=dtype, device=dev)
        self.v_cache = torch.zeros((B, L, H, d), dtype=dtype, device=dev)
        self.score = torch.zeros((B, L), dtype=f32, device=dev)
        self.start = torch.zeros((B,), dtype=i32, device=dev)
        self._score0 = torch.zeros((B, L), dtype=f32, device=dev)
        self._score0[:, :prompt] = float("inf")
        self._start0 = torch.full((B,), prompt, dtype=i32, device=dev)
        # buffers sized for the widest window (all L rows); a step over Lw rows
        # uses the first B * Lw rows of each as a contiguous [B, Lw, ...] view
        self._cos = torch.empty((B * L,), dtype=f32, device=dev)
        self._idx = torch.empty((B * L,), dtype=i32, device=dev)
        self.o = torch.empty((B, row_cap, H, d), dtype=dtype, device=dev)
        self.lse = torch.empty((B, H, row_cap), dtype=f32, device=dev)
        self.count = torch.zeros((B,), dtype=i32, device=dev)
        self.colsum = torch.empty((B, H, L), dtype=f32, device=dev)
        self.argmax = torch.zeros((B, L), dtype=i32, device=dev)
        self.margin = torch.zeros((B, L), dtype=f32, device=dev)
        self.length = torch.zeros((B,), dtype=i32, device=dev)
        self.dev_status = torch.zeros((1,), dtype=i32, device=dev)
        cw = _lib.dllm_confidence_workspace_bytes(B, L, V, dtype)
        self.conf_ws = torch.empty((max(cw, 16),), dtype=torch.uint8, device=dev)
        self._side = torch.cuda.Stream(dev)
        self._fork = torch.cuda.Event()
        self._join = torch.cuda.Event()
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        self.attn_ws = None
        if 2 * B * H < sms:
            aw = _lib.dllm_attention_workspace_bytes(B, L, H, d, row_cap, dtype)
            self.attn_ws = torch.empty((max(aw, 16),), dtype=torch.uint8, device=dev)

    # ------------------------------------------------------------------ views
    def cos(self, Lw: int) -> torch.Tensor:
        return self._cos[:self.B * Lw].view(self.B, Lw)

    def idx(self, Lw: int) -> torch.Tensor:
        return self._idx[:self.B * Lw].view(self.B, Lw)

    # ------------------------------------------------------------------ state
    def reset(self, k_cache: torch.Tensor, v_cache: torch.Tensor):
        """Start a new sequence on the current stream: the given cache, then
        reset_positions()."""
        self.k_cache.copy_(k_cache, non_blocking=True)
        self.v_cache.copy_(v_cache, non_blocking=True)
        self.reset_positions()

    def reset_positions(self):
        """score and start of a new sequence, copied on the current stream
        from device-resident initial values (two device-to-device copies, no
        kernel): score 0 on the generated positions (no prediction yet), +inf
        on the prompt (committed); start = prompt.  The cache is left as it
        is."""
        self.score.copy_(self._score0, non_blocking=True)
        self.start.copy_(self._start0, non_blocking=True)

    # ------------------------------------------------------------------ step
    def step(self, cur: torch.Tensor, prev: torch.Tensor, q: torch.Tensor,
             k_new: torch.Tensor, v_new: torch.Tensor, logits: torch.Tensor, win_start: int,
             events: Optional[Sequence[torch.cuda.Event]] = None, stream=None):
        """Launch one partial step over the window [win_start, L).

        ``cur``/``prev`` [B, L, D] hidden states (only the window's rows are
        read); ``k_new``/``v_new`` [B, Lw, H, d] and ``q`` [B, row_cap, H,
        d], row i the fresh row of the i-th active position; ``logits``
        [B, R, V] (R <= row_cap rows allocated), row r the logits of the r-th
        active position.  Optional
        ``events`` (7) are recorded on the current stream around the six
        calls (pass ``stream=None`` with them); the calls then run one after
        the other on that stream, the column sums included.  ``stream`` is
        None (the current stream) or a ``torch.cuda.Stream``.
        """
        w = win_start
        Lw = self.L - w
        ev = events
        st = self.dev_status
        idx = self.idx(Lw)
        if ev: ev[0].record()
        _lib.dllm_saliency_select(cur[:, w:], prev[:, w:], self.tau, idx_base=w,
                                  cos_out=self.cos(Lw), idx_out=idx, count_out=self.count,
                                  dev_status=st, stream=stream)
        if ev: ev[1].record()
        _lib.dllm_kv_scatter(self.k_cache, self.v_cache, k_new, v_new, idx, self.count,
                             dev_status=st, stream=stream)
        if ev: ev[2].record()
        _lib.dllm_partial_attention(q, self.k_cache, self.v_cache, self.count, o_out=self.o,
                                    lse_out=self.lse, with_colsum=False,
                                    ws=False if self.attn_ws is None else self.attn_ws,
                                    dev_status=st, stream=stream)
        if ev:
            ev[3].record()
            _lib.dllm_attention_colsum(q, self.k_cache, self.count, self.lse,
                                       colsum_out=self.colsum, dev_status=st)
            ev[4].record()
        else:  # fork: the column sums on the side stream
            main = torch.cuda.current_stream() if stream is None else stream
            self._fork.record(main)
            self._side.wait_event(self._fork)
            _lib.dllm_attention_colsum(q, self.k_cache, self.count, self.lse,
                                       colsum_out=self.colsum, dev_status=st, stream=self._side)
        _lib.dllm_confidence(logits, R_max=Lw, count=self.count, out_idx=idx, out_cols=self.L,
                             conf_out=self.score, argmax_out=self.argmax,
                             margin_out=self.margin, ws=self.conf_ws, dev_status=st,
                             stream=stream)
        if ev: ev[5].record()
        _lib.dllm_stable_prefix(self.score, self.start, self.tau_c, min_commit=True,
                                advance_start=True, len_out=self.length, dev_status=st,
                                stream=stream)
        if ev:
            ev[6].record()
        else:  # join
            self._join.record(self._side)
            main.wait_event(self._join)
        return self
