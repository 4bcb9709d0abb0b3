"""Partial denoising step for masked-diffusion language models on B300.

One step recomputes only a selected subset of token positions: cosine saliency
selection, KV-cache scatter, partial attention with column sums, confidence /
argmax / margin, and the longest stable prefix; around it the lock criterion
between steps, the adaptive prefix threshold, the stable rows' output update,
the attention-guided decoding order and the slow/fast phase controller.  Every operation runs in the
hand-written sm_103a kernels of ``libdllm.so`` behind a C ABI
(``include/dllm.h``); the functions below are its ctypes binding, with the
same names.  PyTorch provides device memory and streams only.
"""
from ._lib import (  # noqa: F401
    DllmError,
    LIB_PATH,
    SIGNATURES,
    SlowFast,
    SlowFastDevice,
    dllm_adaptive_prefix,
    dllm_approx_attention_update,
    dllm_attention_colsum,
    dllm_attn_sampler_select,
    dllm_attn_scores,
    dllm_attention_workspace_bytes,
    dllm_confidence,
    dllm_confidence_workspace_bytes,
    dllm_kv_scatter,
    dllm_lock_criterion,
    dllm_lock_criterion_conf,
    dllm_lock_workspace_bytes,
    dllm_partial_attention,
    dllm_read_stream,
    dllm_saliency_select,
    dllm_slowfast_select,
    dllm_snap_prefix,
    dllm_stable_prefix,
    dllm_version,
    load_library,
)
from .loop import BlockDecodeLoop  # noqa: F401
from .step import PartialStep  # noqa: F401
