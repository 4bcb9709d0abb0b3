"""Float64 CPU oracle of the partial denoising step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, calls or links anything here and shares no
code with it.

Every function is the plain definition of one output, written in numpy float64
on dtype-decoded inputs, and cites the page passage it follows.  Pins that tie
it to something other than itself live in ``tests/test_oracle_pins.py``.
"""
from .dllm_oracle import (  # noqa: F401
    saliency_cos,
    salient_flags,
    compact,
    saliency_select,
    confidence,
    kv_scatter,
    partial_attention,
    stable_prefix,
    lock_kl,
    lock_decision,
    adaptive_prefix,
    approx_attention_update,
    attn_scores,
    attn_sampler_select,
    slowfast_phases,
    slowfast_fast_select,
    slowfast_slow_select,
    slowfast_select,
    snap_prefix,
    step,
)
