"""dllm_confidence_static_ws: the confidence entry point that allocates nothing.

Some callers cannot allocate device memory: a plugin that its host framework
hands only raw input and output pointers, or a latency-critical caller that
cannot pay for cudaMalloc's device-wide synchronisation.  For them the
library offers a variant of dllm_confidence whose scratch is a fixed-size
array defined in device memory by the library itself.  This test calls it
through the C ABI and checks its outputs against the workspace version and
against the float64 oracle on two calls in a row (the second on different
inputs, so stale scratch contents from the first call would show), and that a
shape needing more scratch than the stated maximum, or a NULL argument, is
refused before anything is launched.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

STATIC_WS_BYTES = 4 << 20  # DLLM_CONFIDENCE_STATIC_WS_BYTES in include/dllm.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from partial_attention_saliency_b300 import build
    build.build_library()
    from partial_attention_saliency_b300 import _lib
    return _lib.load_library()


def _static_ws_call(lib, logits, R_max, row_idx, count, out_cols, st):
    B, R_src, V = logits.shape
    dev = logits.device
    conf = torch.full((B, out_cols), -1.0, device=dev)
    am = torch.full((B, out_cols), -1, dtype=torch.int32, device=dev)
    mg = torch.full((B, out_cols), -1.0, device=dev)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.dllm_confidence_static_ws(
        p(logits), 1, B, R_src, V, logits.stride(1), logits.stride(0), R_max, p(row_idx),
        p(count), None, out_cols, p(conf), p(am), p(mg), p(st),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.dllm_last_error()
    return conf, am, mg


def _workspace_call(logits, R_max, row_idx, count, out_cols):
    import partial_attention_saliency_b300 as dl
    B = logits.shape[0]
    dev = logits.device
    conf = torch.full((B, out_cols), -1.0, device=dev)
    am = torch.full((B, out_cols), -1, dtype=torch.int32, device=dev)
    mg = torch.full((B, out_cols), -1.0, device=dev)
    dl.dllm_confidence(logits, R_max=R_max, row_idx=row_idx, count=count, out_cols=out_cols,
                       conf_out=conf, argmax_out=am, margin_out=mg)
    return conf, am, mg


def _same(a, b):
    (ca, aa, ma), (cb, ab, mb) = a, b
    ca, cb = ca.double().cpu().numpy(), cb.double().cpu().numpy()
    assert np.array_equal(aa.cpu().numpy(), ab.cpu().numpy())
    assert np.all(np.abs(ca - cb) <= 1e-6 + 1e-4 * np.abs(cb))
    assert np.max(np.abs(ma.double().cpu().numpy() - mb.double().cpu().numpy())) <= 1e-6


def _oracle_check(got, logits, count=None, row_idx=None):
    conf, am, mg = (t.cpu() for t in got)
    z = logits.double().cpu().numpy()
    rc, ra, rm = oracle.confidence(z, count=None if count is None else count.cpu().numpy(),
                                   row_idx=None if row_idx is None else row_idx.cpu().numpy())
    n = rc.shape[1] if count is None else None
    for b in range(z.shape[0]):
        k = n if count is None else int(count[b])
        c = conf[b, :k].double().numpy()
        assert np.all(np.abs(c - rc[b, :k]) <= 1e-6 + 1e-4 * np.abs(rc[b, :k]))
        assert np.array_equal(am[b, :k].numpy(), ra[b, :k])
        assert np.max(np.abs(mg[b, :k].double().numpy() - rm[b, :k]), initial=0.0) <= 1e-6


def test_static_scratch_matches_workspace_version_two_calls(lib):
    dev = torch.device("cuda")
    st = torch.zeros((1,), dtype=torch.int32, device=dev)
    # call 1: one row per generated position of the 1K step, vocabulary 126464
    g = torch.Generator().manual_seed(101)
    s = workloads.STEP_1K
    logits1 = workloads.normal(g, (1, s.logit_rows, s.V), 2.0, torch.bfloat16).to(dev)
    got = _static_ws_call(lib, logits1, s.logit_rows, None, None, s.logit_rows, st)
    torch.cuda.synchronize()
    _same(got, _workspace_call(logits1, s.logit_rows, None, None, s.logit_rows))
    _oracle_check(got, logits1)
    # call 2: other inputs, gathered rows and device counts
    logits2 = workloads.normal(g, (3, 64, 40000), 2.0, torch.bfloat16).to(dev)
    row_idx = torch.randint(0, 64, (3, 48), generator=g, dtype=torch.int32).to(dev)
    count = torch.tensor([48, 7, 0], dtype=torch.int32, device=dev)
    got = _static_ws_call(lib, logits2, 48, row_idx, count, 48, st)
    torch.cuda.synchronize()
    _same(got, _workspace_call(logits2, 48, row_idx, count, 48))
    _oracle_check(got, logits2, count=count, row_idx=row_idx)
    assert int(st[0]) == 0


def test_static_scratch_rejects_oversize_before_launch(lib):
    need = lib.dllm_confidence_workspace_bytes(1, 65536, 126464, 1)
    assert need > STATIC_WS_BYTES
    dummy = ctypes.c_void_p(0x1000)  # never dereferenced: the size check comes first
    rc = lib.dllm_confidence_static_ws(dummy, 1, 1, 65536, 126464, 126464, 0, 65536, None, None,
                                       None, 65536, dummy, dummy, None, None, None)
    assert rc == 1
    assert b"static maximum" in lib.dllm_last_error()
    # a NULL argument is refused before the scratch is looked up
    rc = lib.dllm_confidence_static_ws(None, 1, 1, 8, 1000, 1000, 0, 8, None, None, None, 8,
                                       dummy, dummy, None, None, None)
    assert rc == 1
