"""The C-ABI library loads and exports what include/dllm.h declares.

No GPU needed: only host-side entry points run (version, workspace queries and
argument validation, which returns before any CUDA call).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    with open(os.path.join(ROOT, "include", "dllm.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dllm_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from partial_attention_saliency_b300 import build
    path = build.build_library()
    from partial_attention_saliency_b300 import _lib
    return _lib.load_library(path)


def test_header_declares_the_five_entry_points():
    names = _declared_functions()
    for n in ("dllm_saliency_select", "dllm_confidence", "dllm_kv_scatter",
              "dllm_partial_attention", "dllm_stable_prefix"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from partial_attention_saliency_b300 import _lib
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"
    assert set(_lib.SIGNATURES) <= set(_declared_functions())


def test_version_and_no_error(lib):
    assert lib.dllm_version().decode().startswith("dllm ")
    assert "sm_103a" in lib.dllm_version().decode()


def test_workspace_queries_host_only(lib):
    assert lib.dllm_confidence_workspace_bytes(1, 512, 126464, 1) > 0
    assert lib.dllm_confidence_workspace_bytes(0, 512, 126464, 1) == 0
    assert lib.dllm_confidence_workspace_bytes(1, 512, 126464, 7) == 0
    # grows with rows
    a = lib.dllm_confidence_workspace_bytes(1, 100, 126464, 1)
    b = lib.dllm_confidence_workspace_bytes(2, 100, 126464, 1)
    assert b == 2 * a


def test_invalid_arguments_rejected_before_launch(lib):
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    st = lib.dllm_saliency_select(None, p, 1, 1, 8, 8, 8, 64, None, 0.99, 0, p, p, p, None, None)
    assert st == 1 and b"NULL" in lib.dllm_last_error()
    st = lib.dllm_saliency_select(p, p, 1, 1, 8, 8, 4, 64, None, 0.99, 0, p, p, p, None, None)
    assert st == 1 and b"row_stride" in lib.dllm_last_error()
    st = lib.dllm_saliency_select(p, p, 9, 1, 8, 8, 8, 64, None, 0.99, 0, p, p, p, None, None)
    assert st == 1 and b"dtype" in lib.dllm_last_error()
    st = lib.dllm_confidence(p, 1, 1, 4, 1, 1, 4, 4, None, None, None, 4, p, p, None, p, 1 << 20,
                             None, None)
    assert st == 1 and b"V=1" in lib.dllm_last_error()
    st = lib.dllm_confidence(p, 1, 1, 4, 64, 64, 256, 4, None, None, None, 4, p, p, None, p, 0,
                             None, None)
    assert st == 1 and b"workspace" in lib.dllm_last_error()
    st = lib.dllm_partial_attention(p, p, p, 1, 1, 16, 2, 48, 8, p, 0.0, p, p, None, None, 0,
                                    None, None)
    assert st == 2 and b"head dim" in lib.dllm_last_error()
    st = lib.dllm_partial_attention(p, p, p, 1, 1, 16, 2, 128, 8, p, 0.0, p, None, p, None, 0,
                                    None, None)
    assert st == 1 and b"lse" in lib.dllm_last_error()
    st = lib.dllm_kv_scatter(p, p, p, None, 1, 1, 16, 2, 128, 8, p, p, None, None)
    assert st == 1
    st = lib.dllm_stable_prefix(p, 0, 16, p, 0.9, 1, 0, p, None, None)
    assert st == 1


def test_lock_workspace_query_host_only(lib):
    # one 32-byte partial per (row, chunk of 256 threads x 4 16-byte vectors)
    assert lib.dllm_lock_workspace_bytes(1, 100, 126464, 1) == 100 * 16 * 32
    assert lib.dllm_lock_workspace_bytes(2, 100, 126464, 1) == 2 * 100 * 16 * 32
    assert lib.dllm_lock_workspace_bytes(1, 100, 126464, 0) == 100 * 31 * 32  # f32: 4 per vector
    assert lib.dllm_lock_workspace_bytes(0, 100, 126464, 1) == 0
    assert lib.dllm_lock_workspace_bytes(1, 100, 126464, 5) == 0


def test_lock_and_adaptive_prefix_rejected_before_launch(lib):
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    big = 1 << 30

    def lock(z=p, V=64, rs=64, R_max=4, out_cols=4, kl=p, locked=None, ws_bytes=big, ws=p,
             row_idx=None):
        return lib.dllm_lock_criterion(z, p, 1, 1, 4, V, rs, 4 * rs, R_max, row_idx, None, None,
                                       out_cols, 0.1, 0.5, kl, p, locked, ws, ws_bytes, None,
                                       None)

    assert lock(z=None) == 1 and b"NULL" in lib.dllm_last_error()
    assert lock(kl=None) == 1 and b"NULL" in lib.dllm_last_error()
    assert lock(V=0) == 1
    assert lock(rs=32) == 1 and b"row_stride" in lib.dllm_last_error()
    assert lock(R_max=8) == 1 and b"row_idx" in lib.dllm_last_error()
    assert lock(R_max=8, row_idx=p, out_cols=4) == 1 and b"out_cols" in lib.dllm_last_error()
    assert lock(ws_bytes=16) == 1 and b"workspace" in lib.dllm_last_error()
    assert lock(ws=ctypes.c_void_p(0x1004)) == 1 and b"misaligned" in lib.dllm_last_error()
    st = lib.dllm_lock_criterion(p, p, 1, 1, 4, 64, 64, 256, 20000, p, None, p, 20000, 0.1, 0.5,
                                 p, p, p, p, big, None, None)
    assert st == 1 and b"16384" in lib.dllm_last_error()

    def lock_conf(conf=p, am=p, V=64, rs=64):
        return lib.dllm_lock_criterion_conf(p, p, 1, 1, 4, V, rs, 4 * rs, 4, None, None, None, 4,
                                            0.1, 0.5, p, p, conf, am, None, None, p, big, None,
                                            None)

    assert lock_conf(conf=None) == 1 and b"conf_out" in lib.dllm_last_error()
    assert lock_conf(am=None) == 1 and b"argmax_out" in lib.dllm_last_error()
    assert lock_conf(V=1, rs=1) == 1 and b"V=1" in lib.dllm_last_error()
    assert lock_conf(rs=32) == 1 and b"row_stride" in lib.dllm_last_error()
    st = lib.dllm_adaptive_prefix(None, 1, 16, p, 0.25, 0.5, 0, p, p, None, None)
    assert st == 1 and b"NULL" in lib.dllm_last_error()
    st = lib.dllm_adaptive_prefix(p, 1, 16, p, 0.25, 1.5, 0, p, p, None, None)
    assert st == 1 and b"fractions" in lib.dllm_last_error()
    st = lib.dllm_adaptive_prefix(p, 0, 16, p, 0.25, 0.5, 0, p, p, None, None)
    assert st == 1


def test_sampler_and_stable_row_update_rejected_before_launch(lib):
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    assert lib.dllm_attn_scores(None, 1, 32, 16, 0, p, None, None) == 1
    assert lib.dllm_attn_scores(p, 1, 0, 16, 0, p, None, None) == 1
    st = lib.dllm_attn_sampler_select(p, 1, 16385, None, 0.0, 0.0, 0, p, p, None, None)
    assert st == 1 and b"16384" in lib.dllm_last_error()
    st = lib.dllm_attn_sampler_select(p, 1, 16, None, float("nan"), 0.0, 0, p, p, None, None)
    assert st == 1 and b"NaN" in lib.dllm_last_error()

    def upd(d=128, o=p, B=1):
        return lib.dllm_approx_attention_update(p, p, p, p, p, 1, B, 64, 2, d, 8, p, p, 8, p, p,
                                                0.0, o, None, None)

    assert upd(o=None) == 1 and b"NULL" in lib.dllm_last_error()
    assert upd(d=48) == 2 and b"head dim" in lib.dllm_last_error()
    assert upd(B=0) == 1


def test_diagnostics_rejected_before_launch(lib):
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    assert lib.dllm_set_wait_limit(-1) == 1
    assert lib.dllm_exp2_fma_eval(None, p, 4, None) == 1
    assert lib.dllm_read_stream(None, 4096, p, p, None) == 1
    assert lib.dllm_read_stream(p, 4100, p, p, None) == 1  # not a multiple of 16
    assert b"multiple of 16" in lib.dllm_last_error()
    assert lib.dllm_read_stream(ctypes.c_void_p(0x1008), 4096, p, p, None) == 1  # misaligned
    assert lib.dllm_read_stream(p, 4096, None, p, None) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    from partial_attention_saliency_b300 import _lib
    with pytest.raises(ImportError):
        saved = _lib._LIB
        _lib._LIB = None
        try:
            _lib.load_library(str(tmp_path / "missing.so"))
        finally:
            _lib._LIB = saved


def test_every_kernel_waits_for_its_predecessor():
    # Every kernel is launched with programmatic dependent launch, so it may
    # be resident while the previous kernel on the stream still runs; it must
    # execute pdl_wait() before touching global memory.  Static check of the
    # sources: each __global__ body starts with pdl_wait(), and no launch
    # bypasses launch_pdl (or launch_serial, the same launch without early
    # residency, where pdl_wait() returns at once).
    src_dir = os.path.join(ROOT, "partial_attention_saliency_b300", "csrc")
    kernels = 0
    for name in sorted(os.listdir(src_dir)):
        if not name.endswith(".cu"):
            continue
        with open(os.path.join(src_dir, name)) as f:
            text = f.read()
        assert "<<<" not in text, f"{name}: kernel launched without launch_pdl"
        for m in re.finditer(r"__global__[^{;]*\{", text):
            body = text[m.end():m.end() + 120].strip()
            assert body.startswith("pdl_wait();"), f"{name}: kernel body does not start with pdl_wait()"
            kernels += 1
    assert kernels >= 12
