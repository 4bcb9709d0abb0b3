"""The library's own machinery on the GPU: the FMA-pipe exponential against
its error bound, a bounded pipeline wait that runs out, and the read-stream
reference kernel reading every chunk it is given.

Bounded waits: every mbarrier wait of the kernels gives up after a limit,
records DLLM_ERR_TIMEOUT in dev_status, drains the kernel's own copies and
tensor-core work and returns.  dllm_set_wait_limit shortens that limit to a
single clock cycle, so the first wait that does not succeed at once runs
out; the attention call must then return with TIMEOUT in dev_status, and the
next call with the default limit must be correct again (nothing left
behind).  (The streaming confidence kernel takes the same limit, but its
waits complete within the hardware's own suspend time of a single try-wait,
so no limit makes them run out.)  The
waits only get shorter: nothing is made to hang or fault.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

DLLM_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def dl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from partial_attention_saliency_b300 import build
    build.build_library()
    import partial_attention_saliency_b300 as dl
    dl.load_library()
    return dl


def test_exp2_fma_within_bound(dl):
    lib = dl.load_library()
    x = torch.linspace(-125.0, 128.0, 4_000_001, dtype=torch.float64).float()
    x = torch.cat([x, torch.arange(-125, 129, dtype=torch.float32), torch.tensor([-200.0, -125.5])])
    xd = x.cuda()
    y = torch.empty_like(xd)
    assert lib.dllm_exp2_fma_eval(ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                                  xd.numel(), None) == 0
    torch.cuda.synchronize()
    got = y.double().cpu().numpy()
    xs = np.maximum(x.double().numpy(), -125.0)  # clamped at -125
    rel = np.abs(got / np.exp2(xs) - 1.0)
    assert rel.max() <= 2.7e-6, (rel.max(), xs[rel.argmax()])


def _with_limit(lib, cycles, fn):
    assert lib.dllm_set_wait_limit(cycles) == 0
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        assert lib.dllm_set_wait_limit(0) == 0


def test_attention_wait_runs_out_and_next_call_is_clean(dl):
    lib = dl.load_library()
    B, L, H, M = 2, 1024, 8, 200
    g = torch.Generator().manual_seed(5)
    q = workloads.normal(g, (B, M, H, 128), 1.0, torch.bfloat16)
    k = workloads.normal(g, (B, L, H, 128), 1.0, torch.bfloat16)
    v = workloads.normal(g, (B, L, H, 128), 1.0, torch.bfloat16)
    count = torch.tensor([M, 77], dtype=torch.int32)
    qd, kd, vd, cd = q.cuda(), k.cuda(), v.cuda(), count.cuda()
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    _with_limit(lib, 1, lambda: dl.dllm_partial_attention(qd, kd, vd, cd, with_colsum=False,
                                                           dev_status=st))
    assert int(st[0]) == DLLM_ERR_TIMEOUT
    st.zero_()
    o, lse, cs = dl.dllm_partial_attention(qd, kd, vd, cd, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    f = lambda t: t.double().numpy()  # noqa: E731
    for b, h in ((0, 0), (1, 5)):
        n = int(count[b])
        ro, rl, rcs = oracle.partial_attention(f(q)[b:b + 1, :, h:h + 1], f(k)[b:b + 1, :, h:h + 1],
                                               f(v)[b:b + 1, :, h:h + 1], [n])
        go = o[b, :n, h].double().cpu().numpy()
        assert np.all(np.abs(go - ro[0, :n, 0]) <= 2e-2 + 1e-2 * np.abs(ro[0, :n, 0]))
        assert np.max(np.abs(cs[b, h].double().cpu().numpy() - rcs[0, 0])) <= 1e-4


@pytest.mark.parametrize("nbytes", [16, 32768 * 3 + 4096, 64 << 20])
def test_read_stream_reads_each_chunk(dl, nbytes):
    # chunk c (32 KB, the last one shorter) is the (c // grid)-th chunk of CTA
    # c % grid, which adds its byte at offset ((c // grid) % 16) * 16 (0 when
    # the chunk is shorter than that) into the sink
    g = torch.Generator().manual_seed(nbytes)
    buf = torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8)
    sink = torch.zeros((1,), dtype=torch.int32, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    dl.dllm_read_stream(buf.cuda(), nbytes, sink, dev_status=st)
    torch.cuda.synchronize()
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    nch = (nbytes + 32767) // 32768
    c = np.arange(nch)
    size = np.minimum(nbytes - c * 32768, 32768)
    off = ((c // grid) % 16) * 16
    off = np.where(off < size, off, 0)
    want = int(buf.numpy()[c * 32768 + off].astype(np.int64).sum())
    assert int(st[0]) == 0
    assert int(sink[0]) == want
