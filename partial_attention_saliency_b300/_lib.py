"""ctypes binding of libdllm.so: argument marshalling only.

Every wrapper takes torch CUDA tensors, checks dtypes/devices/strides, passes
raw device pointers and the current CUDA stream to the C entry point of the
same name, and raises ``DllmError`` on a non-zero status.  No computation of
the step happens here: it all runs in the library's kernels.  If the library
is missing the import fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libdllm.so")

DLLM_OK = 0
STATUS_NAMES = {0: "DLLM_OK", 1: "DLLM_ERR_INVALID_ARG", 2: "DLLM_ERR_UNSUPPORTED",
                3: "DLLM_ERR_CUDA", 4: "DLLM_ERR_DEVICE_CHECK", 5: "DLLM_ERR_TIMEOUT"}
DTYPES = {torch.float32: 0, torch.bfloat16: 1}

# Every symbol include/dllm.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
SIGNATURES = {
    "dllm_version": (ctypes.c_char_p, []),
    "dllm_last_error": (ctypes.c_char_p, []),
    "dllm_saliency_select": (_I, [_P, _P, _I, _I, _I, _I, _I64, _I64, _P, _F, ctypes.c_int32,
                                  _P, _P, _P, _P, _P]),
    "dllm_confidence_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "dllm_confidence": (_I, [_P, _I, _I, _I, _I, _I64, _I64, _I, _P, _P, _P, _I, _P, _P, _P,
                             _P, _SZ, _P, _P]),
    "dllm_confidence_static_ws": (_I, [_P, _I, _I, _I, _I, _I64, _I64, _I, _P, _P, _P, _I, _P,
                                       _P, _P, _P, _P]),
    "dllm_kv_scatter": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "dllm_attention_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "dllm_partial_attention": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _F, _P, _P, _P, _P,
                                    _SZ, _P, _P]),
    "dllm_attention_colsum": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _F, _P, _P, _P, _P]),
    "dllm_stable_prefix": (_I, [_P, _I, _I, _P, _F, _I, _I, _P, _P, _P]),
    "dllm_lock_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "dllm_lock_criterion": (_I, [_P, _P, _I, _I, _I, _I, _I64, _I64, _I, _P, _P, _P, _I, _F, _F,
                                 _P, _P, _P, _P, _SZ, _P, _P]),
    "dllm_lock_criterion_conf": (_I, [_P, _P, _I, _I, _I, _I, _I64, _I64, _I, _P, _P, _P, _I, _F,
                                      _F, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "dllm_adaptive_prefix": (_I, [_P, _I, _I, _P, _F, _F, _I, _P, _P, _P, _P]),
    "dllm_attn_scores": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "dllm_attn_sampler_select": (_I, [_P, _I, _I, _P, _F, _F, _I, _P, _P, _P, _P]),
    "dllm_approx_attention_update": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P,
                                          _I, _P, _P, _F, _P, _P, _P]),
    "dllm_snap_prefix": (_I, [_P, _I, _I, _I, _P, _P, _P, _I, _P, _P]),
    "dllm_slowfast_create": (_I, [_I, _I, ctypes.c_double, ctypes.POINTER(_P)]),
    "dllm_slowfast_observe": (_I, [_P, _P, _P, _P, _P]),
    "dllm_slowfast_destroy": (None, [_P]),
    "dllm_slowfast_state_bytes": (_SZ, [_I, _I]),
    "dllm_exp2_fma_eval": (_I, [_P, _P, _I, _P]),
    "dllm_set_wait_limit": (_I, [ctypes.c_longlong]),
    "dllm_read_stream": (_I, [_P, _SZ, _P, _P, _P]),
    "dllm_slowfast_observe_device": (_I, [_P, _I, _I, ctypes.c_double, _P, _P, _P, _P, _P, _P]),
    "dllm_slowfast_select": (_I, [_P, _P, _I, _I, _P, _P, _P, _F, _I, _I, _P, _P, _P, _P]),
}


class DllmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_LIB: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdllm.so (once) and declare every exported entry point."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m partial_attention_saliency_b300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(status: int):
    if status != DLLM_OK:
        raise DllmError(status, load_library().dllm_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype(*ts: torch.Tensor) -> int:
    dt = ts[0].dtype
    for t in ts:
        if t.dtype != dt:
            raise TypeError(f"dtype mismatch: {t.dtype} vs {dt}")
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")
    if dt not in DTYPES:
        raise TypeError(f"unsupported dtype {dt}; use float32 or bfloat16")
    return DTYPES[dt]


def _need(t: torch.Tensor, dtype, shape, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: need contiguous CUDA {dtype} {tuple(shape)}, got "
                         f"{t.dtype} {tuple(t.shape)} contiguous={t.is_contiguous()}")


def dllm_version() -> str:
    return load_library().dllm_version().decode()


def dllm_confidence_workspace_bytes(B: int, R_max: int, V: int, dtype: torch.dtype) -> int:
    return int(load_library().dllm_confidence_workspace_bytes(B, R_max, V, DTYPES[dtype]))


def dllm_attention_workspace_bytes(B: int, L: int, H: int, d: int, M_max: int,
                                   dtype: torch.dtype) -> int:
    return int(load_library().dllm_attention_workspace_bytes(B, L, H, d, M_max, DTYPES[dtype]))


def dllm_saliency_select(cur: torch.Tensor, prev: torch.Tensor, tau: float, *,
                         locked: Optional[torch.Tensor] = None, idx_base: int = 0,
                         cos_out=None, idx_out=None, count_out=None, dev_status=None,
                         stream=None):
    """Cosine saliency + ordered compaction over a [B, Lw, D] window.

    ``cur``/``prev`` may be strided views (last dim contiguous).  Returns
    (cos [B, Lw] f32, idx [B, Lw] i32, count [B] i32).
    """
    lib = load_library()
    dt = _dtype(cur, prev)
    if cur.dim() != 3 or cur.shape != prev.shape or cur.stride() != prev.stride():
        raise ValueError("cur/prev must be [B, Lw, D] with identical strides")
    if cur.stride(2) != 1:
        raise ValueError("the hidden dim must be contiguous")
    B, Lw, D = cur.shape
    dev = cur.device
    cos_out = torch.empty((B, Lw), dtype=torch.float32, device=dev) if cos_out is None else cos_out
    idx_out = torch.empty((B, Lw), dtype=torch.int32, device=dev) if idx_out is None else idx_out
    count_out = torch.empty((B,), dtype=torch.int32, device=dev) if count_out is None else count_out
    _need(cos_out, torch.float32, (B, Lw), "cos_out")
    _need(idx_out, torch.int32, (B, Lw), "idx_out")
    _need(count_out, torch.int32, (B,), "count_out")
    if locked is not None:
        _need(locked, torch.uint8, (B, Lw), "locked")
    _check(lib.dllm_saliency_select(_ptr(cur), _ptr(prev), dt, B, Lw, D, cur.stride(1),
                                    cur.stride(0), _ptr(locked), float(tau), int(idx_base),
                                    _ptr(cos_out), _ptr(idx_out), _ptr(count_out),
                                    _ptr(dev_status), _stream(stream)))
    return cos_out, idx_out, count_out


def dllm_confidence(logits: torch.Tensor, *, R_max: Optional[int] = None, row_idx=None,
                    count=None, out_idx=None, out_cols: Optional[int] = None, conf_out=None,
                    argmax_out=None, margin_out=None, with_margin: bool = True, ws=None,
                    dev_status=None, stream=None):
    """Confidence, argmax and margin per logit row.

    ``logits`` [B, R_src, V] (last dim contiguous, rows may be strided).
    Outputs are [B, out_cols] (default out_cols = R_max).  Returns
    (conf, argmax, margin-or-None).
    """
    lib = load_library()
    dt = _dtype(logits)
    if logits.dim() != 3 or logits.stride(2) != 1:
        raise ValueError("logits must be [B, R_src, V] with a contiguous vocabulary dim")
    B, R_src, V = logits.shape
    R_max = R_src if R_max is None else int(R_max)
    out_cols = R_max if out_cols is None else int(out_cols)
    dev = logits.device
    if conf_out is None:
        conf_out = torch.empty((B, out_cols), dtype=torch.float32, device=dev)
    if argmax_out is None:
        argmax_out = torch.empty((B, out_cols), dtype=torch.int32, device=dev)
    if margin_out is None and with_margin:
        margin_out = torch.empty((B, out_cols), dtype=torch.float32, device=dev)
    for t, n, ty in ((conf_out, "conf_out", torch.float32), (argmax_out, "argmax_out", torch.int32),
                     (margin_out, "margin_out", torch.float32)):
        if t is not None and (t.dtype != ty or not t.is_cuda or t.stride(-1) != 1
                              or t.shape[0] != B or (B > 1 and t.stride(0) != out_cols)):
            raise ValueError(f"{n}: need CUDA {ty} [B, out_cols] rows")
    for t, n in ((row_idx, "row_idx"), (out_idx, "out_idx")):
        if t is not None:
            _need(t, torch.int32, (B, R_max), n)
    if count is not None:
        _need(count, torch.int32, (B,), "count")
    need = lib.dllm_confidence_workspace_bytes(B, R_max, V, dt)
    if ws is None:
        ws = torch.empty((max(int(need), 16),), dtype=torch.uint8, device=dev)
    _check(lib.dllm_confidence(_ptr(logits), dt, B, R_src, V, logits.stride(1), logits.stride(0),
                               R_max, _ptr(row_idx), _ptr(count), _ptr(out_idx), out_cols,
                               _ptr(conf_out), _ptr(argmax_out), _ptr(margin_out), _ptr(ws),
                               ws.numel() * ws.element_size(), _ptr(dev_status),
                               _stream(stream)))
    return conf_out, argmax_out, margin_out


def dllm_kv_scatter(k_cache, v_cache, k_new, v_new, idx, count, *, dev_status=None, stream=None):
    """Write fresh K/V rows into the cache in place at idx[b, :count[b]]."""
    lib = load_library()
    dt = _dtype(k_cache, v_cache, k_new, v_new)
    B, L, H, d = k_cache.shape
    M_max = k_new.shape[1]
    _need(k_cache, k_cache.dtype, (B, L, H, d), "k_cache")
    _need(v_cache, k_cache.dtype, (B, L, H, d), "v_cache")
    _need(k_new, k_cache.dtype, (B, M_max, H, d), "k_new")
    _need(v_new, k_cache.dtype, (B, M_max, H, d), "v_new")
    _need(idx, torch.int32, (B, M_max), "idx")
    _need(count, torch.int32, (B,), "count")
    _check(lib.dllm_kv_scatter(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), dt, B, L,
                               H, d, M_max, _ptr(idx), _ptr(count), _ptr(dev_status),
                               _stream(stream)))
    return k_cache, v_cache


def dllm_partial_attention(q, k_cache, v_cache, count, *, scale: float = 0.0, o_out=None,
                           lse_out=None, colsum_out=None, with_lse: bool = True,
                           with_colsum: bool = True, ws=None, dev_status=None, stream=None):
    """Attention of the active query rows over the whole cache (+ column sums).

    ``ws``: the workspace for key-range splits; None allocates one, False
    passes none (the key range is then never split and no merge runs).
    Returns (o [B, M_max, H, d], lse [B, H, M_max] or None, colsum [B, H, L] or None).
    """
    lib = load_library()
    dt = _dtype(q, k_cache, v_cache)
    B, M_max, H, d = q.shape
    L = k_cache.shape[1]
    _need(q, q.dtype, (B, M_max, H, d), "q")
    _need(k_cache, q.dtype, (B, L, H, d), "k_cache")
    _need(v_cache, q.dtype, (B, L, H, d), "v_cache")
    _need(count, torch.int32, (B,), "count")
    dev = q.device
    o_out = torch.empty_like(q) if o_out is None else o_out
    if lse_out is None and (with_lse or with_colsum):
        lse_out = torch.empty((B, H, M_max), dtype=torch.float32, device=dev)
    if colsum_out is None and with_colsum:
        colsum_out = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    _need(o_out, q.dtype, (B, M_max, H, d), "o_out")
    if lse_out is not None:
        _need(lse_out, torch.float32, (B, H, M_max), "lse_out")
    if colsum_out is not None:
        _need(colsum_out, torch.float32, (B, H, L), "colsum_out")
    need = int(lib.dllm_attention_workspace_bytes(B, L, H, d, M_max, dt))
    if ws is None and need > 0:  # the workspace is optional: without it no key-range split
        ws = torch.empty((need,), dtype=torch.uint8, device=dev)
    if ws is False:
        ws = None
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.dllm_partial_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), dt, B, L, H, d,
                                      M_max, _ptr(count), float(scale), _ptr(o_out),
                                      _ptr(lse_out), _ptr(colsum_out), _ptr(ws), ws_bytes,
                                      _ptr(dev_status), _stream(stream)))
    return o_out, lse_out, colsum_out


def dllm_attention_colsum(q, k_cache, count, lse, *, scale: float = 0.0, colsum_out=None,
                          dev_status=None, stream=None):
    """Per-key column sums over the active rows from a given lse.

    Returns colsum [B, H, L] f32.
    """
    lib = load_library()
    dt = _dtype(q, k_cache)
    B, M_max, H, d = q.shape
    L = k_cache.shape[1]
    _need(q, q.dtype, (B, M_max, H, d), "q")
    _need(k_cache, q.dtype, (B, L, H, d), "k_cache")
    _need(count, torch.int32, (B,), "count")
    _need(lse, torch.float32, (B, H, M_max), "lse")
    if colsum_out is None:
        colsum_out = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    _need(colsum_out, torch.float32, (B, H, L), "colsum_out")
    _check(lib.dllm_attention_colsum(_ptr(q), _ptr(k_cache), dt, B, L, H, d, M_max, _ptr(count),
                                     float(scale), _ptr(lse), _ptr(colsum_out), _ptr(dev_status),
                                     _stream(stream)))
    return colsum_out


def dllm_stable_prefix(score, start, tau: float, *, min_commit: bool = True,
                       advance_start: bool = False, len_out=None, dev_status=None, stream=None):
    """Longest stable prefix per batch row; optionally advances ``start`` in place."""
    lib = load_library()
    B, L = score.shape
    _need(score, torch.float32, (B, L), "score")
    _need(start, torch.int32, (B,), "start")
    len_out = torch.empty((B,), dtype=torch.int32, device=score.device) if len_out is None else len_out
    _need(len_out, torch.int32, (B,), "len_out")
    _check(lib.dllm_stable_prefix(_ptr(score), B, L, _ptr(start), float(tau), int(min_commit),
                                  int(advance_start), _ptr(len_out), _ptr(dev_status),
                                  _stream(stream)))
    return len_out


def dllm_lock_workspace_bytes(B: int, R_max: int, V: int, dtype: torch.dtype) -> int:
    return int(load_library().dllm_lock_workspace_bytes(B, R_max, V, DTYPES[dtype]))


def dllm_lock_criterion(logits_cur, logits_prev, eps: float, *, gate_q: float = 0.0,
                        R_max: Optional[int] = None, row_idx=None, count=None, out_idx=None,
                        out_cols: Optional[int] = None, kl_out=None, unc_out=None,
                        locked_inout=None, ws=None, dev_status=None, stream=None):
    """Local KL divergence between two steps, uncertainty and lock flags.

    ``logits_cur``/``logits_prev`` [B, R_src, V] with identical strides.
    Returns (kl [B, out_cols], unc [B, out_cols], locked_inout or None).
    """
    return _lock_call(False, logits_cur, logits_prev, eps, gate_q, R_max, row_idx, count,
                      out_idx, out_cols, kl_out, unc_out, None, None, None, locked_inout, ws,
                      dev_status, stream)[:3]


def dllm_lock_criterion_conf(logits_cur, logits_prev, eps: float, *, gate_q: float = 0.0,
                             R_max: Optional[int] = None, row_idx=None, count=None,
                             out_idx=None, out_cols: Optional[int] = None, kl_out=None,
                             unc_out=None, conf_out=None, argmax_out=None, margin_out=None,
                             with_margin: bool = True, locked_inout=None, ws=None,
                             dev_status=None, stream=None):
    """dllm_lock_criterion plus the current rows' confidence, argmax and
    margin (dllm_confidence's outputs) from one read of the logits.
    Returns (kl, unc, locked_inout or None, conf, argmax, margin or None)."""
    if margin_out is None and with_margin and logits_cur.dim() == 3:
        B = logits_cur.shape[0]
        cols = (logits_cur.shape[1] if R_max is None else int(R_max)) if out_cols is None \
            else int(out_cols)
        margin_out = torch.empty((B, cols), dtype=torch.float32, device=logits_cur.device)
    return _lock_call(True, logits_cur, logits_prev, eps, gate_q, R_max, row_idx, count,
                      out_idx, out_cols, kl_out, unc_out, conf_out, argmax_out, margin_out,
                      locked_inout, ws, dev_status, stream)


def _lock_call(conf: bool, logits_cur, logits_prev, eps, gate_q, R_max, row_idx, count, out_idx,
               out_cols, kl_out, unc_out, conf_out, argmax_out, margin_out, locked_inout, ws,
               dev_status, stream):
    lib = load_library()
    dt = _dtype(logits_cur, logits_prev)
    if logits_cur.dim() != 3 or logits_cur.shape != logits_prev.shape \
            or logits_cur.stride() != logits_prev.stride() or logits_cur.stride(2) != 1:
        raise ValueError("logits must be [B, R_src, V] with identical strides, vocabulary contiguous")
    B, R_src, V = logits_cur.shape
    R_max = R_src if R_max is None else int(R_max)
    out_cols = R_max if out_cols is None else int(out_cols)
    dev = logits_cur.device
    kl_out = torch.empty((B, out_cols), dtype=torch.float32, device=dev) if kl_out is None else kl_out
    unc_out = torch.empty((B, out_cols), dtype=torch.float32, device=dev) if unc_out is None else unc_out
    _need(kl_out, torch.float32, (B, out_cols), "kl_out")
    _need(unc_out, torch.float32, (B, out_cols), "unc_out")
    if conf:
        if conf_out is None:
            conf_out = torch.empty((B, out_cols), dtype=torch.float32, device=dev)
        if argmax_out is None:
            argmax_out = torch.empty((B, out_cols), dtype=torch.int32, device=dev)
        _need(conf_out, torch.float32, (B, out_cols), "conf_out")
        _need(argmax_out, torch.int32, (B, out_cols), "argmax_out")
        if margin_out is not None:
            _need(margin_out, torch.float32, (B, out_cols), "margin_out")
    if locked_inout is not None:
        _need(locked_inout, torch.uint8, (B, out_cols), "locked_inout")
    for t, n in ((row_idx, "row_idx"), (out_idx, "out_idx")):
        if t is not None:
            _need(t, torch.int32, (B, R_max), n)
    if count is not None:
        _need(count, torch.int32, (B,), "count")
    need = lib.dllm_lock_workspace_bytes(B, R_max, V, dt)
    if ws is None:
        ws = torch.empty((max(int(need), 16),), dtype=torch.uint8, device=dev)
    common = (_ptr(logits_cur), _ptr(logits_prev), dt, B, R_src, V, logits_cur.stride(1),
              logits_cur.stride(0), R_max, _ptr(row_idx), _ptr(count), _ptr(out_idx), out_cols,
              float(eps), float(gate_q), _ptr(kl_out), _ptr(unc_out))
    tail = (_ptr(locked_inout), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status),
            _stream(stream))
    if conf:
        _check(lib.dllm_lock_criterion_conf(*common, _ptr(conf_out), _ptr(argmax_out),
                                            _ptr(margin_out), *tail))
    else:
        _check(lib.dllm_lock_criterion(*common, *tail))
    return kl_out, unc_out, locked_inout, conf_out, argmax_out, margin_out


def dllm_adaptive_prefix(score, start, lo: float, hi: float, *, advance_start: bool = False,
                         len_out=None, tau_out=None, dev_status=None, stream=None):
    """Longest stable prefix whose threshold adapts to a fraction [lo, hi] of
    the active length.  Returns (len [B] int32, tau [B] float32)."""
    lib = load_library()
    B, L = score.shape
    _need(score, torch.float32, (B, L), "score")
    _need(start, torch.int32, (B,), "start")
    dev = score.device
    len_out = torch.empty((B,), dtype=torch.int32, device=dev) if len_out is None else len_out
    tau_out = torch.empty((B,), dtype=torch.float32, device=dev) if tau_out is None else tau_out
    _need(len_out, torch.int32, (B,), "len_out")
    _need(tau_out, torch.float32, (B,), "tau_out")
    _check(lib.dllm_adaptive_prefix(_ptr(score), B, L, _ptr(start), float(lo), float(hi),
                                    int(advance_start), _ptr(len_out), _ptr(tau_out),
                                    _ptr(dev_status), _stream(stream)))
    return len_out, tau_out


def dllm_attn_scores(colsum, *, score_inout=None, accumulate: bool = False, dev_status=None,
                     stream=None):
    """Sum over heads of the attention column sums ``colsum`` [B, H, L];
    ``accumulate`` adds onto ``score_inout`` (layers).  Returns [B, L]."""
    lib = load_library()
    B, H, L = colsum.shape
    _need(colsum, torch.float32, (B, H, L), "colsum")
    if score_inout is None:
        if accumulate:
            raise ValueError("accumulate needs score_inout")
        score_inout = torch.empty((B, L), dtype=torch.float32, device=colsum.device)
    _need(score_inout, torch.float32, (B, L), "score_inout")
    _check(lib.dllm_attn_scores(_ptr(colsum), B, H, L, int(accumulate), _ptr(score_inout),
                                _ptr(dev_status), _stream(stream)))
    return score_inout


def dllm_attn_sampler_select(score, *, candidates=None, tau: float = 0.0, gamma: float = 0.0,
                             k_max: int = 0, order_out=None, n_out=None, dev_status=None,
                             stream=None):
    """Candidates by descending score and how many of them to decode.
    Returns (order [B, L] int32, n [B] int32)."""
    lib = load_library()
    B, L = score.shape
    _need(score, torch.float32, (B, L), "score")
    if candidates is not None:
        _need(candidates, torch.uint8, (B, L), "candidates")
    dev = score.device
    order_out = torch.empty((B, L), dtype=torch.int32, device=dev) if order_out is None else order_out
    n_out = torch.empty((B,), dtype=torch.int32, device=dev) if n_out is None else n_out
    _need(order_out, torch.int32, (B, L), "order_out")
    _need(n_out, torch.int32, (B,), "n_out")
    _check(lib.dllm_attn_sampler_select(_ptr(score), B, L, _ptr(candidates), float(tau),
                                        float(gamma), int(k_max), _ptr(order_out), _ptr(n_out),
                                        _ptr(dev_status), _stream(stream)))
    return order_out, n_out


def dllm_approx_attention_update(q_prev, lse_prev, k_prev, v_prev, v_new, idx, count, stable_idx,
                                 stable_count, o_inout, *, scale: float = 0.0, dev_status=None,
                                 stream=None):
    """Update the outputs ``o_inout`` [B, L, H, d] of the stable rows in place
    from the value changes of the salient rows.  Returns ``o_inout``."""
    lib = load_library()
    dt = _dtype(q_prev, k_prev, v_prev, v_new, o_inout)
    B, L, H, d = q_prev.shape
    M_max = v_new.shape[1]
    N_max = stable_idx.shape[1]
    for t, n in ((q_prev, "q_prev"), (k_prev, "k_prev"), (v_prev, "v_prev"), (o_inout, "o_inout")):
        _need(t, q_prev.dtype, (B, L, H, d), n)
    _need(v_new, q_prev.dtype, (B, M_max, H, d), "v_new")
    _need(lse_prev, torch.float32, (B, H, L), "lse_prev")
    _need(idx, torch.int32, (B, M_max), "idx")
    _need(count, torch.int32, (B,), "count")
    _need(stable_idx, torch.int32, (B, N_max), "stable_idx")
    _need(stable_count, torch.int32, (B,), "stable_count")
    _check(lib.dllm_approx_attention_update(_ptr(q_prev), _ptr(lse_prev), _ptr(k_prev),
                                            _ptr(v_prev), _ptr(v_new), dt, B, L, H, d, M_max,
                                            _ptr(idx), _ptr(count), N_max, _ptr(stable_idx),
                                            _ptr(stable_count), float(scale), _ptr(o_inout),
                                            _ptr(dev_status), _stream(stream)))
    return o_inout


def dllm_snap_prefix(tokens, delim, start, len_inout, *, min_len: int = 1, dev_status=None,
                     stream=None):
    """Snap the committed blocks [start, start + len) to their last boundary
    token (``delim`` [V] uint8 flags); ``len_inout`` [B] is updated in place
    and returned."""
    lib = load_library()
    B, L = tokens.shape
    V = delim.shape[0]
    _need(tokens, torch.int32, (B, L), "tokens")
    _need(delim, torch.uint8, (V,), "delim")
    _need(start, torch.int32, (B,), "start")
    _need(len_inout, torch.int32, (B,), "len_inout")
    _check(lib.dllm_snap_prefix(_ptr(tokens), B, L, V, _ptr(delim), _ptr(start), _ptr(len_inout),
                                int(min_len), _ptr(dev_status), _stream(stream)))
    return len_inout


class SlowFast:
    """Host-side SlowFast phase controller (``dllm_slowfast_*``).

    ``observe(start, e_cand)`` takes [B] int32 host arrays (numpy or CPU
    tensors) of this step and returns (phase [B], region_end [B]) as int32
    numpy arrays: phase 1 with the region [start, region_end) on a fast step.
    """

    def __init__(self, B: int, window: int, sigma2_stable: float):
        import numpy as np
        self._np = np
        self._lib = load_library()
        self.B = int(B)
        h = _P()
        _check(self._lib.dllm_slowfast_create(self.B, int(window), float(sigma2_stable),
                                              ctypes.byref(h)))
        self._h = h

    def observe(self, start, e_cand):
        np = self._np
        s = np.ascontiguousarray(np.asarray(start, dtype=np.int32))
        e = np.ascontiguousarray(np.asarray(e_cand, dtype=np.int32))
        if s.shape != (self.B,) or e.shape != (self.B,):
            raise ValueError(f"start and e_cand must be [{self.B}]")
        phase = np.zeros(self.B, dtype=np.int32)
        end = np.zeros(self.B, dtype=np.int32)
        _check(self._lib.dllm_slowfast_observe(self._h, s.ctypes.data, e.ctypes.data,
                                               phase.ctypes.data, end.ctypes.data))
        return phase, end

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.dllm_slowfast_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()


class SlowFastDevice:
    """Device-side SlowFast phase controller (``dllm_slowfast_observe_device``):
    its state and per-step arrays live on the device, so a decoding loop
    reads nothing back.  ``observe(start, pred_len)`` takes [B] int32 CUDA
    tensors (e_cand = start + pred_len) and returns (phase, region_end), [B]
    int32 CUDA tensors written in place on every call."""

    def __init__(self, B: int, window: int, sigma2_stable: float, device=None):
        lib = load_library()
        self.B, self.window, self.sigma2 = int(B), int(window), float(sigma2_stable)
        n = int(lib.dllm_slowfast_state_bytes(self.B, self.window)) // 4
        dev = torch.device("cuda") if device is None else device
        self.state = torch.zeros((n,), dtype=torch.int32, device=dev)
        self.phase = torch.zeros((self.B,), dtype=torch.int32, device=dev)
        self.region_end = torch.zeros((self.B,), dtype=torch.int32, device=dev)

    def reset(self):
        self.state.zero_()

    def observe(self, start, pred_len, *, dev_status=None, stream=None):
        _need(start, torch.int32, (self.B,), "start")
        _need(pred_len, torch.int32, (self.B,), "pred_len")
        _check(load_library().dllm_slowfast_observe_device(
            _ptr(self.state), self.B, self.window, self.sigma2, _ptr(start), _ptr(pred_len),
            _ptr(self.phase), _ptr(self.region_end), _ptr(dev_status), _stream(stream)))
        return self.phase, self.region_end


def dllm_slowfast_select(conf, start, phase, region_end, tau_high: float, width: int, k: int, *,
                         masked=None, idx_out=None, count_out=None, dev_status=None,
                         stream=None):
    """The positions a SlowFast step unmasks per batch row (fast phase: the
    masked region positions above tau_high; slow phase: the k most confident
    masked positions of [start, start + width)).  Returns (idx [B, L] int32
    ascending then -1, count [B] int32)."""
    lib = load_library()
    B, L = conf.shape
    _need(conf, torch.float32, (B, L), "conf")
    for t, n in ((start, "start"), (phase, "phase"), (region_end, "region_end")):
        _need(t, torch.int32, (B,), n)
    if masked is not None:
        _need(masked, torch.uint8, (B, L), "masked")
    dev = conf.device
    idx_out = torch.empty((B, L), dtype=torch.int32, device=dev) if idx_out is None else idx_out
    count_out = torch.empty((B,), dtype=torch.int32, device=dev) if count_out is None else count_out
    _need(idx_out, torch.int32, (B, L), "idx_out")
    _need(count_out, torch.int32, (B,), "count_out")
    _check(lib.dllm_slowfast_select(_ptr(conf), _ptr(masked), B, L, _ptr(start), _ptr(phase),
                                    _ptr(region_end), float(tau_high), int(width), int(k),
                                    _ptr(idx_out), _ptr(count_out), _ptr(dev_status),
                                    _stream(stream)))
    return idx_out, count_out


def dllm_read_stream(buf, nbytes: int, sink, *, dev_status, stream=None):
    """Reads the first ``nbytes`` bytes of ``buf`` (a contiguous device
    tensor) once, in one launch that does nothing else: the reference time of
    a read-bound launch of that size.  ``sink`` int32 [1] accumulates a byte
    of every 32 KB chunk; ``dev_status`` int32 [1]."""
    if not buf.is_contiguous() or nbytes > buf.numel() * buf.element_size():
        raise ValueError("dllm_read_stream: buf must be contiguous and hold nbytes")
    _need(sink, torch.int32, (1,), "sink")
    _need(dev_status, torch.int32, (1,), "dev_status")
    _check(load_library().dllm_read_stream(_ptr(buf), int(nbytes), _ptr(sink), _ptr(dev_status),
                                           _stream(stream)))
