"""GPU parity: every entry point through the C ABI against the float64 oracle.

Inputs come from the seeded generators in ``workloads``; expected values come
from ``oracle`` only.  Tolerances: bit-exact for indices, counts, argmax,
prefix lengths and cache copies (given the same score arrays); 1e-4 for float32
scores (cos, conf, margin, lse, colsum); max-abs 2e-2 plus rel 1e-2 for
bfloat16 attention outputs; 1e-4 for float32 attention outputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

SCORE_TOL = 1e-4
BF16_ATOL, BF16_RTOL = 2e-2, 1e-2
F32_ATOL = 1e-4


@pytest.fixture(scope="module")
def dl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from partial_attention_saliency_b300 import build
    build.build_library()
    import partial_attention_saliency_b300 as dl
    dl.load_library()
    return dl


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def i32(t):
    return t.detach().cpu().numpy()


def dev(t):
    return t.cuda()


def check_attn(o_gpu, o_ref, dtype, rows_mask=None):
    g, r = f64(o_gpu), o_ref
    if rows_mask is not None:
        g, r = g[rows_mask], r[rows_mask]
    if dtype == torch.bfloat16:
        assert np.all(np.abs(g - r) <= BF16_ATOL + BF16_RTOL * np.abs(r)), np.max(np.abs(g - r))
    else:
        assert np.max(np.abs(g - r)) <= F32_ATOL, np.max(np.abs(g - r))


# ------------------------------------------------------------------ select

def _select_case(dl, inp, tau, win_start, locked=None):
    cur, prev = dev(inp["cur"]), dev(inp["prev"])
    lk = None if locked is None else dev(locked)
    cos, idx, count = dl.dllm_saliency_select(cur[:, win_start:], prev[:, win_start:], tau,
                                              locked=lk, idx_base=win_start)
    torch.cuda.synchronize()
    ref_cos = oracle.saliency_cos(f64(inp["cur"][:, win_start:]), f64(inp["prev"][:, win_start:]))
    assert np.max(np.abs(f64(cos) - ref_cos)) <= SCORE_TOL
    # bit-exact compaction given the GPU's own cosines
    ref_idx, ref_count = oracle.compact(
        oracle.salient_flags(i32(cos), tau, None if locked is None else locked.numpy()), win_start)
    assert np.array_equal(i32(count), ref_count)
    assert np.array_equal(i32(idx), ref_idx)
    return cos, idx, count


def test_select_tiny_f32_planted(dl):
    s = workloads.TINY_F32
    inp = workloads.make_step(s)
    _, idx, count = _select_case(dl, inp, s.tau, 0)
    assert i32(idx)[0, : int(count[0])].tolist() == inp["planted"][0].tolist()


def test_select_1k_window_planted(dl):
    s = workloads.STEP_1K
    inp = workloads.make_step(s, with_logits=False)
    _, idx, count = _select_case(dl, inp, s.tau, s.win_start)
    assert int(count[0]) == s.n_salient
    assert i32(idx)[0, : s.n_salient].tolist() == inp["planted"][0].tolist()


@pytest.mark.parametrize("frac,pattern", [(0.05, "random"), (0.5, "cluster")])
def test_select_batch8_full_size(dl, frac, pattern):
    s = workloads.BATCH8_2K
    n = round(frac * s.L)
    inp = workloads.make_step(s, n_salient=n, pattern=pattern, with_logits=False, m_max=1)
    _, idx, count = _select_case(dl, inp, s.tau, 0)
    for b in range(s.B):
        assert i32(idx)[b, : int(count[b])].tolist() == inp["planted"][b].tolist()


def test_select_ragged_strided_locked_edges(dl):
    g = torch.Generator().manual_seed(5)
    B, L, D = 3, 5000, 77  # D not a multiple of the vector width, Lw > one compaction chunk
    big = torch.randn((B, L, D + 5), generator=g, dtype=torch.float64)
    cur = big[:, :, :D].to(torch.bfloat16)
    prev = (big[:, :, :D] + 0.2 * torch.randn((B, L, D), generator=g, dtype=torch.float64)).to(torch.bfloat16)
    cur_d = dev(torch.randn((B, L, D + 5), dtype=torch.bfloat16))
    cur_d[:, :, :D] = dev(cur)
    prev_d = dev(torch.randn((B, L, D + 5), dtype=torch.bfloat16))
    prev_d[:, :, :D] = dev(prev)
    cur_v, prev_v = cur_d[:, :, :D], prev_d[:, :, :D]  # row stride D + 5
    locked = (torch.rand((B, L), generator=g) < 0.3).to(torch.uint8)
    for tau in (0.99, 0.98, 2.0, -2.0):
        cos, idx, count = dl.dllm_saliency_select(cur_v, prev_v, tau, locked=dev(locked), idx_base=3)
        torch.cuda.synchronize()
        ref_cos = oracle.saliency_cos(f64(cur), f64(prev))
        assert np.max(np.abs(f64(cos) - ref_cos)) <= SCORE_TOL
        ref_idx, ref_count = oracle.compact(oracle.salient_flags(i32(cos), tau, locked.numpy()), 3)
        assert np.array_equal(i32(count), ref_count)
        assert np.array_equal(i32(idx), ref_idx)
    # zero vectors: both zero -> 1, one zero -> 0 (so salient at tau 0.99)
    z = torch.zeros((1, 4, 64), dtype=torch.float32)
    a = torch.ones((1, 4, 64), dtype=torch.float32)
    cos, idx, count = dl.dllm_saliency_select(dev(torch.cat([z[:, :2], a[:, :2]], 1)),
                                              dev(torch.cat([z[:, :1], a[:, :1], z[:, :1], a[:, :1]], 1)), 0.99)
    assert f64(cos).tolist() == [[1.0, 0.0, 0.0, 1.0]]
    assert i32(count).tolist() == [2] and i32(idx).tolist() == [[1, 2, -1, -1]]


# ------------------------------------------------------------------ confidence

def _conf_compare(conf, am, mg, rc, ra, rm):
    assert np.array_equal(am, ra)
    assert np.all(np.abs(conf - rc) <= 1e-6 + SCORE_TOL * np.abs(rc)), np.max(np.abs(conf - rc) / rc)
    assert np.max(np.abs(mg - rm)) <= 1e-6


def test_confidence_tiny_f32(dl):
    s = workloads.TINY_F32
    inp = workloads.make_step(s)
    conf, am, mg = dl.dllm_confidence(dev(inp["logits"]))
    torch.cuda.synchronize()
    rc, ra, rm = oracle.confidence(f64(inp["logits"]))
    _conf_compare(f64(conf), i32(am), f64(mg), rc, ra, rm)


def test_confidence_1k_full_size(dl):
    s = workloads.STEP_1K
    g = torch.Generator().manual_seed(s.seed)
    logits = workloads.normal(g, (1, s.logit_rows, s.V), 2.0, s.dtype)
    conf, am, mg = dl.dllm_confidence(dev(logits))
    torch.cuda.synchronize()
    rc, ra, rm = oracle.confidence(f64(logits))
    _conf_compare(f64(conf), i32(am), f64(mg), rc, ra, rm)


def test_confidence_repeated_calls_reuse_buffers(dl):
    # Back-to-back calls on the same workspace and outputs with different
    # logits: each call's merge must see only that call's partial results
    # (no stale data from the previous call on the same addresses).
    s = workloads.STEP_1K
    R = 256
    ws = torch.empty((dl.dllm_confidence_workspace_bytes(1, R, s.V, s.dtype),), dtype=torch.uint8,
                     device="cuda")
    conf = torch.empty((1, R), device="cuda")
    am = torch.empty((1, R), dtype=torch.int32, device="cuda")
    mg = torch.empty((1, R), device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    for seed in (11, 12, 13):
        g = torch.Generator().manual_seed(seed)
        logits = workloads.normal(g, (1, R, s.V), 2.0, s.dtype)
        dl.dllm_confidence(dev(logits), conf_out=conf, argmax_out=am, margin_out=mg, ws=ws,
                           dev_status=st)
        torch.cuda.synchronize()
        rc, ra, rm = oracle.confidence(f64(logits))
        _conf_compare(f64(conf), i32(am), f64(mg), rc, ra, rm)
    assert int(st[0]) == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V", [2, 7, 1001, 16384, 40000])
def test_confidence_ragged_vocab_and_ties(dl, dtype, V):
    g = torch.Generator().manual_seed(V)
    z = torch.round(torch.randn((2, 9, V), generator=g, dtype=torch.float64) * 4) / 4
    z[0, 3, V // 2] = 50.0
    z[0, 3, V - 1] = 50.0  # tie: lowest index wins, margin 0
    z = z.to(dtype)
    conf, am, mg = dl.dllm_confidence(dev(z))
    torch.cuda.synchronize()
    rc, ra, rm = oracle.confidence(f64(z))
    _conf_compare(f64(conf), i32(am), f64(mg), rc, ra, rm)
    if V // 2 != V - 1:
        assert i32(am)[0, 3] == V // 2 and f64(mg)[0, 3] == 0.0


@pytest.mark.parametrize("B,R,V,counts", [
    (3, 40, 126464, [40, 0, 17]),   # ragged counts, an empty batch row
    (2, 9, 300000, None),           # 10 chunks of 64 KB per row
    (65, 3, 1000, None),            # more batch rows than the streaming kernel stages counts for
])
def test_confidence_kernel_paths(dl, B, R, V, counts):
    # the streaming kernel and the merge on aligned rows: rows past a count
    # are not written, every other row matches the oracle
    g = torch.Generator().manual_seed(V + B)
    z = workloads.normal(g, (B, R, V), 2.0, torch.bfloat16)
    cnt = None if counts is None else torch.tensor(counts, dtype=torch.int32)
    st = dev(torch.zeros((1,), dtype=torch.int32))
    conf = dev(torch.full((B, R), -7.0))
    am = dev(torch.full((B, R), -7, dtype=torch.int32))
    mg = dev(torch.full((B, R), -7.0))
    dl.dllm_confidence(dev(z), count=None if cnt is None else dev(cnt), conf_out=conf,
                       argmax_out=am, margin_out=mg, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    rc, ra, rm = oracle.confidence(f64(z), count=None if cnt is None else cnt.numpy())
    for b in range(B):
        n = R if cnt is None else int(cnt[b])
        if n > 0:
            _conf_compare(f64(conf)[b:b + 1, :n], i32(am)[b:b + 1, :n], f64(mg)[b:b + 1, :n],
                          rc[b:b + 1, :n], ra[b:b + 1, :n], rm[b:b + 1, :n])
        assert np.all(f64(conf)[b, n:] == -7.0)  # rows past the count are not written


def test_confidence_strided_rows_row_idx_count_out_idx(dl):
    g = torch.Generator().manual_seed(11)
    B, R_src, V = 2, 20, 3000
    base = torch.randn((B, R_src, V + 8), generator=g, dtype=torch.float64).to(torch.bfloat16)
    z = dev(base)[:, :, :V]  # row stride V + 8
    R_max = 6
    row_idx = torch.tensor([[19, 0, 7, 7, 3, 1], [2, 4, 6, 8, 10, 12]], dtype=torch.int32)
    count = torch.tensor([4, 6], dtype=torch.int32)
    out_idx = torch.tensor([[30, 2, 11, 12, 0, 0], [0, 5, 9, 13, 21, 39]], dtype=torch.int32)
    out_cols = 40
    conf = dev(torch.full((B, out_cols), -7.0))
    am = dev(torch.full((B, out_cols), -7, dtype=torch.int32))
    mg = dev(torch.full((B, out_cols), -7.0))
    dl.dllm_confidence(z, R_max=R_max, row_idx=dev(row_idx), count=dev(count),
                       out_idx=dev(out_idx), out_cols=out_cols, conf_out=conf, argmax_out=am,
                       margin_out=mg)
    torch.cuda.synchronize()
    rc, ra, rm = oracle.confidence(f64(base[:, :, :V]), count=count.numpy(), row_idx=row_idx.numpy())
    ec = np.full((B, out_cols), -7.0)
    ea = np.full((B, out_cols), -7, dtype=np.int32)
    em = np.full((B, out_cols), -7.0)
    for b in range(B):
        for r in range(int(count[b])):
            c = int(out_idx[b, r])
            ec[b, c], ea[b, c], em[b, c] = rc[b, r], ra[b, r], rm[b, r]
    _conf_compare(f64(conf), i32(am), f64(mg), ec, ea, em)


# ------------------------------------------------------------------ scatter

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_kv_scatter_bit_exact(dl, dtype):
    s = workloads.BATCH8_2K
    B, L, H, d, M = 4, 600, 8, 128, 300
    g = torch.Generator().manual_seed(3)
    kc = workloads.normal(g, (B, L, H, d), 1.0, dtype)
    vc = workloads.normal(g, (B, L, H, d), 1.0, dtype)
    kn = workloads.normal(g, (B, M, H, d), 1.0, dtype)
    vn = workloads.normal(g, (B, M, H, d), 1.0, dtype)
    idx = torch.full((B, M), -1, dtype=torch.int32)
    counts = [0, 1, 37, M]
    for b, c in enumerate(counts):
        pos = torch.sort(torch.randperm(L, generator=g)[:c]).values if c < L else torch.arange(L)
        if b == 2:  # a contiguous run (prefix append)
            pos = torch.arange(100, 100 + c)
        idx[b, :c] = pos.to(torch.int32)
    count = torch.tensor(counts, dtype=torch.int32)
    kd, vd = dev(kc), dev(vc)
    dl.dllm_kv_scatter(kd, vd, dev(kn), dev(vn), dev(idx), dev(count))
    torch.cuda.synchronize()
    rk, rv = oracle.kv_scatter(kc.numpy() if dtype == torch.float32 else kc.view(torch.int16).numpy(),
                               vc.numpy() if dtype == torch.float32 else vc.view(torch.int16).numpy(),
                               kn.numpy() if dtype == torch.float32 else kn.view(torch.int16).numpy(),
                               vn.numpy() if dtype == torch.float32 else vn.view(torch.int16).numpy(),
                               idx.numpy(), count.numpy())
    gk = kd.cpu() if dtype == torch.float32 else kd.cpu().view(torch.int16)
    gv = vd.cpu() if dtype == torch.float32 else vd.cpu().view(torch.int16)
    assert np.array_equal(gk.numpy(), rk) and np.array_equal(gv.numpy(), rv)


def test_kv_scatter_bad_indices_flag_status(dl):
    B, L, H, d, M = 1, 32, 2, 32, 4
    kc = dev(torch.zeros((B, L, H, d), dtype=torch.bfloat16))
    vc = dev(torch.zeros((B, L, H, d), dtype=torch.bfloat16))
    kn = dev(torch.ones((B, M, H, d), dtype=torch.bfloat16))
    vn = dev(torch.ones((B, M, H, d), dtype=torch.bfloat16))
    st = dev(torch.zeros((1,), dtype=torch.int32))
    # row 1 goes backwards, row 2 is out of range, row 3 is below its predecessor (40)
    idx = dev(torch.tensor([[3, 2, 40, 5]], dtype=torch.int32))
    dl.dllm_kv_scatter(kc, vc, kn, vn, idx, dev(torch.tensor([4], dtype=torch.int32)), dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 4  # DLLM_ERR_DEVICE_CHECK
    written = (kc.float().abs().sum((2, 3)) > 0).cpu().numpy()[0]
    assert written[3] and not written[2] and not written[5]
    st.zero_()
    dl.dllm_kv_scatter(kc, vc, kn, vn, idx, dev(torch.tensor([9], dtype=torch.int32)), dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 4


# ------------------------------------------------------------------ attention

def _attn_case(dl, B, M_max, counts, L, H, d, dtype, seed=0, scale=0.0, colsum=True):
    g = torch.Generator().manual_seed(seed)
    q = workloads.normal(g, (B, M_max, H, d), 1.0, dtype)
    k = workloads.normal(g, (B, L, H, d), 1.0, dtype)
    v = workloads.normal(g, (B, L, H, d), 1.0, dtype)
    count = torch.tensor(counts, dtype=torch.int32)
    o, lse, cs = dl.dllm_partial_attention(dev(q), dev(k), dev(v), dev(count), scale=scale,
                                           with_colsum=colsum)
    torch.cuda.synchronize()
    ro, rl, rc = oracle.partial_attention(f64(q), f64(k), f64(v), counts,
                                          None if scale <= 0 else scale)
    mask = np.zeros((B, M_max), dtype=bool)
    for b, c in enumerate(counts):
        mask[b, :c] = True
    check_attn(o, ro, dtype, mask)
    gl = f64(lse)
    for b, c in enumerate(counts):
        assert np.max(np.abs(gl[b, :, :c] - rl[b, :, :c]), initial=0) <= SCORE_TOL
    if colsum:
        assert np.max(np.abs(f64(cs) - rc)) <= SCORE_TOL
    return o, lse, cs


def test_attention_tiny_f32(dl):
    _attn_case(dl, 1, 64, [16], 64, 2, 32, torch.float32)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_attention_f32_ragged(dl, d):
    _attn_case(dl, 2, 40, [33, 7], 71, 3, d, torch.float32, seed=d)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_attention_bf16_ragged(dl, d):
    _attn_case(dl, 2, 300, [130, 257], 333, 4, d, torch.bfloat16, seed=d + 1)


def test_attention_bf16_edges(dl):
    # count 0 (colsum all zero), count M_max, one key, explicit scale
    _, _, cs = _attn_case(dl, 3, 128, [0, 128, 5], 1, 2, 128, torch.bfloat16, seed=4)
    assert np.all(f64(cs)[0] == 0)
    _attn_case(dl, 1, 256, [200], 513, 2, 128, torch.bfloat16, seed=6, scale=0.05)


def test_attention_1k_full_size(dl):
    s = workloads.STEP_1K
    _attn_case(dl, 1, s.Lw, [s.n_salient], s.L, s.H, s.d, s.dtype, seed=s.seed)


def test_attention_all_active_equals_dense(dl):
    B, L, H, d = 1, 384, 4, 128
    g = torch.Generator().manual_seed(21)
    q = workloads.normal(g, (B, L, H, d), 1.0, torch.bfloat16)
    k = workloads.normal(g, (B, L, H, d), 1.0, torch.bfloat16)
    v = workloads.normal(g, (B, L, H, d), 1.0, torch.bfloat16)
    o, lse, cs = dl.dllm_partial_attention(dev(q), dev(k), dev(v), dev(torch.tensor([L], dtype=torch.int32)))
    torch.cuda.synchronize()
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double().transpose(1, 2), k.double().transpose(1, 2), v.double().transpose(1, 2)).transpose(1, 2)
    check_attn(o, ref.numpy(), torch.bfloat16)
    assert np.allclose(f64(cs).sum(-1), L, atol=1e-4 * L)


def test_attention_batch8_sampled_heads(dl):
    # full 50% size in the launch configuration of the step; oracle on 3 heads
    s = workloads.BATCH8_2K
    M = 1024
    g = torch.Generator().manual_seed(8)
    q = workloads.normal(g, (s.B, M, s.H, s.d), 1.0, s.dtype)
    k = workloads.normal(g, (s.B, s.L, s.H, s.d), 1.0, s.dtype)
    v = workloads.normal(g, (s.B, s.L, s.H, s.d), 1.0, s.dtype)
    counts = [M, 1000, 512, 1, 0, 777, 1024, 100]
    o, lse, cs = dl.dllm_partial_attention(dev(q), dev(k), dev(v), dev(torch.tensor(counts, dtype=torch.int32)))
    torch.cuda.synchronize()
    go, gl, gc = f64(o), f64(lse), f64(cs)
    for b in range(s.B):
        assert abs(gc[b].sum(-1) - counts[b]).max() <= 1e-4 * max(counts[b], 1)
    for b, h in ((0, 0), (5, 17), (7, 31)):
        n = counts[b]
        ro, rl, rc = oracle.partial_attention(f64(q[b:b + 1, :, h:h + 1]), f64(k[b:b + 1, :, h:h + 1]),
                                              f64(v[b:b + 1, :, h:h + 1]), [n])
        check_attn(o[b:b + 1, :n, h:h + 1], ro[:, :n], s.dtype)
        assert np.max(np.abs(gl[b, h, :n] - rl[0, 0, :n])) <= SCORE_TOL
        assert np.max(np.abs(gc[b, h] - rc[0, 0])) <= SCORE_TOL


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 32)])
def test_attention_colsum_call_matches_fused(dl, dtype, d):
    # the column-sum pass as a call of its own reproduces the fused colsum_out
    # bit for bit and matches the oracle
    B, M_max, L, H = 2, 200, 517, 3
    counts = [200, 61]
    g = torch.Generator().manual_seed(31 + d)
    q = workloads.normal(g, (B, M_max, H, d), 1.0, dtype)
    k = workloads.normal(g, (B, L, H, d), 1.0, dtype)
    v = workloads.normal(g, (B, L, H, d), 1.0, dtype)
    cnt = dev(torch.tensor(counts, dtype=torch.int32))
    o, lse, cs = dl.dllm_partial_attention(dev(q), dev(k), dev(v), cnt)
    cs2 = dl.dllm_attention_colsum(dev(q), dev(k), cnt, lse)
    torch.cuda.synchronize()
    assert torch.equal(cs, cs2)
    _, _, rc = oracle.partial_attention(f64(q), f64(k), f64(v), counts)
    assert np.max(np.abs(f64(cs2) - rc)) <= SCORE_TOL


# ------------------------------------------------------------------ stable prefix

def test_stable_prefix_brute_force(dl):
    n = 10
    pats = np.array([[(m >> i) & 1 for i in range(n)] for m in range(1 << n)], dtype=bool)
    score = np.where(pats, 0.95, 0.2).astype(np.float32)
    B = score.shape[0]
    for start_v in (0, 3, n):
        for mc in (False, True):
            start = torch.full((B,), start_v, dtype=torch.int32)
            length = dl.dllm_stable_prefix(dev(torch.from_numpy(score)), dev(start), 0.9, min_commit=mc)
            torch.cuda.synchronize()
            ref = oracle.stable_prefix(score, start.numpy(), 0.9, mc)
            assert np.array_equal(i32(length), ref)


def test_stable_prefix_long_rows_nan_inf_advance(dl):
    g = torch.Generator().manual_seed(2)
    B, L = 5, 4100
    score = torch.full((B, L), float("inf"))
    score[1, 2050] = 0.3
    score[2, :] = torch.rand((L,), generator=g)
    score[3, 77] = float("nan")
    start = torch.tensor([0, 100, 0, 40, L], dtype=torch.int32)
    st_d = dev(start.clone())
    length = dl.dllm_stable_prefix(dev(score), st_d, 0.9, min_commit=True, advance_start=True)
    torch.cuda.synchronize()
    ref = oracle.stable_prefix(score.numpy(), start.numpy(), 0.9, True)
    assert np.array_equal(i32(length), ref)
    assert np.array_equal(i32(st_d), start.numpy() + ref)


# ------------------------------------------------------------------ whole step

def test_step_1k_against_oracle_step(dl):
    s = workloads.STEP_1K
    inp = workloads.make_step(s)
    step = dl.PartialStep(s.B, s.L, s.H, s.d, s.D, s.V, s.dtype, s.win_start, s.logit_rows, s.tau)
    t = {k: dev(inp[k]) for k in ("cur", "prev", "k_cache", "v_cache", "k_new", "v_new", "q")}
    logits = dev(inp["logits"])
    score = dev(torch.full((s.B, s.L), float("inf")))
    start = dev(torch.full((s.B,), s.win_start, dtype=torch.int32))
    step.run(t["cur"], t["prev"], t["k_cache"], t["v_cache"], t["k_new"], t["v_new"], t["q"],
             logits, score, start)
    torch.cuda.synchronize()
    assert int(step.dev_status[0]) == 0
    d = {k: f64(inp[k]) for k in ("cur", "prev", "k_cache", "v_cache", "k_new", "v_new", "q", "logits")}
    ref = oracle.step(d["cur"], d["prev"], d["k_cache"], d["v_cache"], d["k_new"], d["v_new"],
                      d["q"], d["logits"], tau=s.tau, win_start=s.win_start,
                      score=np.full((s.B, s.L), np.inf), start=[s.win_start], tau_c=0.9)
    n = int(step.count[0])
    assert n == s.n_salient
    assert np.array_equal(i32(step.count), ref["count"])
    assert np.array_equal(i32(step.idx), ref["idx"])
    assert np.array_equal(f64(t["k_cache"]), ref["k_cache"])
    check_attn(step.o[:, :n], ref["o"][:, :n], s.dtype)
    assert np.max(np.abs(f64(step.colsum) - ref["colsum"])) <= SCORE_TOL
    gs = f64(score)
    rs = ref["score"]
    w = s.win_start
    assert np.all(np.abs(gs[:, w:] - rs[:, w:]) <= 1e-6 + SCORE_TOL * np.abs(rs[:, w:]))
    assert np.array_equal(i32(step.argmax)[:, w:], ref["argmax"])
    # prefix decision on the GPU's own score array
    assert np.array_equal(i32(step.length), oracle.stable_prefix(gs.astype(np.float32), [w], 0.9, True))


@pytest.mark.parametrize("L,counts", [(1500, [130, 7]), (2100, [1, 260]), (4096, [37])])
def test_attention_split_key_range_ragged(dl, L, counts):
    # few query tiles -> the key range is split across CTAs, then merged
    _attn_case(dl, len(counts), 300, counts, L, 4, 128, torch.bfloat16, seed=L)


def test_attention_without_workspace_matches_split(dl):
    B, M_max, L, H, d = 1, 200, 2048, 8, 128
    g = torch.Generator().manual_seed(77)
    q = dev(workloads.normal(g, (B, M_max, H, d), 1.0, torch.bfloat16))
    k = dev(workloads.normal(g, (B, L, H, d), 1.0, torch.bfloat16))
    v = dev(workloads.normal(g, (B, L, H, d), 1.0, torch.bfloat16))
    count = dev(torch.tensor([150], dtype=torch.int32))
    o1, l1, c1 = dl.dllm_partial_attention(q, k, v, count)  # workspace: split allowed
    no_ws = torch.empty((0,), dtype=torch.uint8, device="cuda")
    o2, l2, c2 = dl.dllm_partial_attention(q, k, v, count, ws=no_ws)  # never split
    torch.cuda.synchronize()
    ro, rl, rc = oracle.partial_attention(f64(q), f64(k), f64(v), [150])
    for o, lse, cs in ((o1, l1, c1), (o2, l2, c2)):
        check_attn(o[:, :150], ro[:, :150], torch.bfloat16)
        assert np.max(np.abs(f64(lse)[:, :, :150] - rl[:, :, :150])) <= SCORE_TOL
        assert np.max(np.abs(f64(cs) - rc)) <= SCORE_TOL


def test_attention_repeatable_run_to_run(dl):
    s = workloads.STEP_1K
    g = torch.Generator().manual_seed(9)
    q = dev(workloads.normal(g, (1, s.Lw, s.H, s.d), 1.0, s.dtype))
    k = dev(workloads.normal(g, (1, s.L, s.H, s.d), 1.0, s.dtype))
    v = dev(workloads.normal(g, (1, s.L, s.H, s.d), 1.0, s.dtype))
    count = dev(torch.tensor([102], dtype=torch.int32))
    a = [t.clone() for t in dl.dllm_partial_attention(q, k, v, count)]
    b = dl.dllm_partial_attention(q, k, v, count)
    torch.cuda.synchronize()
    assert torch.equal(a[0][:, :102], b[0][:, :102])
    assert torch.equal(a[1][:, :, :102], b[1][:, :, :102])
    assert torch.equal(a[2], b[2])


def test_confidence_repeatable_run_to_run(dl):
    g = torch.Generator().manual_seed(19)
    z = dev(workloads.normal(g, (2, 300, 126464), 2.0, torch.bfloat16))
    a = [t.clone() for t in dl.dllm_confidence(z)]
    b = dl.dllm_confidence(z)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_step_repeated_no_bounded_wait_expires(dl):
    # Every pipeline wait in the kernels gives up after about a second and
    # reports DLLM_ERR_TIMEOUT; in normal operation none may expire.  Twenty
    # back-to-back 1K steps must leave dev_status at 0 and finish in well
    # under one expired wait.
    import time
    s = workloads.STEP_1K
    inp = workloads.make_step(s)
    t = {k: dev(inp[k]) for k in ("cur", "prev", "k_cache", "v_cache", "k_new", "v_new", "q",
                                   "logits")}
    step = dl.PartialStep(s.B, s.L, s.H, s.d, s.D, s.V, s.dtype, s.win_start, s.logit_rows,
                          s.tau, device=torch.device("cuda"))
    score = dev(torch.full((s.B, s.L), float("inf")))
    start = dev(torch.full((s.B,), s.win_start, dtype=torch.int32))
    args = (t["cur"], t["prev"], t["k_cache"], t["v_cache"], t["k_new"], t["v_new"], t["q"],
            t["logits"], score, start)
    step.run(*args)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(20):
        step.run(*args)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(step.dev_status[0]) == 0
    assert elapsed < 0.5, elapsed
