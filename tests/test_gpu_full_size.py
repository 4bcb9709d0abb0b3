"""Full-size steps in the launch configuration the bench times, against the oracle.

Two step shapes beyond the 1K step: the long-context step (batch 1, L = 4096,
every unlocked position active, logits of the active rows gathered by row
index and scattered to their positions) and the batch-4 loop step (1024 prompt
+ 1024 generated positions, 134 active per batch row, one logit row per
active row).  Expected values come from the float64 oracle only: selection
and compaction in full (bit-exact, decided on the GPU's own cosines as the
reading of the threshold compare), the cache update bit-exact, attention and
column sums on sampled heads, confidence on every or on sampled active rows,
and the prefix on the GPU's own score array.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

SCORE_TOL = 1e-4
BF16_ATOL, BF16_RTOL = 2e-2, 1e-2


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


def _check_attention_heads(o, lse, cs, q, kc_ref, vc_ref, counts, heads):
    go, gl, gc = f64(o), f64(lse), f64(cs)
    for b, h in heads:
        n = counts[b]
        ro, rl, rc = oracle.partial_attention(q[b:b + 1, :, h:h + 1], kc_ref[b:b + 1, :, h:h + 1],
                                              vc_ref[b:b + 1, :, h:h + 1], [n])
        g = go[b, :n, h]
        r = ro[0, :n, 0]
        assert np.all(np.abs(g - r) <= BF16_ATOL + BF16_RTOL * np.abs(r)), np.max(np.abs(g - r))
        assert np.max(np.abs(gl[b, h, :n] - rl[0, 0, :n])) <= SCORE_TOL
        assert np.max(np.abs(gc[b, h] - rc[0, 0])) <= SCORE_TOL
    for b, n in enumerate(counts):  # every head: column sums add up to the active rows
        assert np.max(np.abs(gc[b].sum(-1) - n)) <= 1e-4 * max(n, 1)


def test_long_context_step_full_size(dl):
    s = workloads.LONG_4K  # tau = 2: every position that is not locked is active
    inp = workloads.make_step(dataclasses.replace(s, logit_rows=0), n_salient=0, with_logits=False)
    g = torch.Generator().manual_seed(41)
    locked = torch.zeros((1, s.L), dtype=torch.uint8)
    locked[0, torch.randperm(s.L, generator=g)[:1229]] = 1  # 30% locked
    R_src = 512
    logits = workloads.normal(g, (1, R_src, s.V), 2.0, s.dtype)
    dev = lambda t: t.cuda()  # noqa: E731
    t = {k: dev(inp[k]) for k in ("cur", "prev", "k_cache", "v_cache", "k_new", "v_new", "q")}
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    cos, idx, count = dl.dllm_saliency_select(t["cur"], t["prev"], s.tau, locked=dev(locked),
                                              dev_status=st)
    dl.dllm_kv_scatter(t["k_cache"], t["v_cache"], t["k_new"], t["v_new"], idx, count,
                       dev_status=st)
    o, lse, cs = dl.dllm_partial_attention(t["q"], t["k_cache"], t["v_cache"], count,
                                           dev_status=st)
    # logits of the active rows: row r reads buffer row idx[r] % 512, and its
    # results land at position idx[r]
    row_idx = (idx.clamp(min=0) % R_src).to(torch.int32).contiguous()
    score = torch.full((1, s.L), float("inf"), device="cuda")
    argmax = torch.full((1, s.L), -1, dtype=torch.int32, device="cuda")
    margin = torch.full((1, s.L), -1.0, device="cuda")
    dl.dllm_confidence(dev(logits), R_max=s.L, row_idx=row_idx, count=count, out_idx=idx,
                       out_cols=s.L, conf_out=score, argmax_out=argmax, margin_out=margin,
                       dev_status=st)
    start = torch.zeros((1,), dtype=torch.int32, device="cuda")
    length = dl.dllm_stable_prefix(score, start, 0.9, min_commit=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0

    # selection: cosines, and bit-exact compaction of the GPU's cosines
    ref_cos = oracle.saliency_cos(f64(inp["cur"]), f64(inp["prev"]))
    assert np.max(np.abs(f64(cos) - ref_cos)) <= SCORE_TOL
    ref_idx, ref_count = oracle.compact(oracle.salient_flags(i32(cos), s.tau, locked.numpy()), 0)
    assert np.array_equal(i32(count), ref_count) and np.array_equal(i32(idx), ref_idx)
    n = int(ref_count[0])
    assert n == s.L - 1229
    # cache update, bit-exact
    kc_ref, vc_ref = oracle.kv_scatter(f64(inp["k_cache"]), f64(inp["v_cache"]), f64(inp["k_new"]),
                                       f64(inp["v_new"]), ref_idx, ref_count)
    assert np.array_equal(f64(t["k_cache"]), kc_ref) and np.array_equal(f64(t["v_cache"]), vc_ref)
    # attention and column sums on sampled heads (all heads for the sums)
    _check_attention_heads(o, lse, cs, f64(inp["q"]), kc_ref, vc_ref, [n],
                           [(0, 0), (0, 13), (0, 31)])
    # confidence on sampled active rows, read back at their positions
    rows = np.linspace(0, n - 1, 48).astype(np.int64)
    pos = ref_idx[0, rows]
    rc, ra, rm = oracle.confidence(f64(logits), count=[len(rows)],
                                   row_idx=(pos % R_src)[None, :])
    gsc = f64(score)[0]
    assert np.all(np.abs(gsc[pos] - rc[0]) <= 1e-6 + SCORE_TOL * np.abs(rc[0]))
    assert np.array_equal(i32(argmax)[0, pos], ra[0])
    assert np.max(np.abs(f64(margin)[0, pos] - rm[0])) <= 1e-6
    locked_pos = np.nonzero(locked.numpy()[0])[0]
    assert np.all(np.isinf(gsc[locked_pos]))  # positions not scored are untouched
    # prefix on the GPU's own score array
    assert np.array_equal(i32(length), oracle.stable_prefix(gsc[None, :].astype(np.float32), [0],
                                                            0.9, True))


def test_batch4_loop_step_full_size(dl):
    s = workloads.LOOP_B4_2K
    n_act = 134
    inp = workloads.make_step(dataclasses.replace(s, logit_rows=0), n_salient=n_act,
                              with_logits=False)
    g = torch.Generator().manual_seed(43)
    rows_made = 160
    logits_rows = workloads.normal(g, (s.B, rows_made, s.V), 2.0, s.dtype)
    logits = torch.zeros((s.B, s.Lw, s.V), dtype=s.dtype, device="cuda")
    logits[:, :rows_made] = logits_rows.cuda()
    w = s.win_start
    t = {k: inp[k].cuda() for k in ("cur", "prev", "k_cache", "v_cache", "k_new", "v_new", "q")}
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    cos, idx, count = dl.dllm_saliency_select(t["cur"][:, w:], t["prev"][:, w:], s.tau,
                                              idx_base=w, dev_status=st)
    dl.dllm_kv_scatter(t["k_cache"], t["v_cache"], t["k_new"], t["v_new"], idx, count,
                       dev_status=st)
    o, lse, cs = dl.dllm_partial_attention(t["q"], t["k_cache"], t["v_cache"], count,
                                           dev_status=st)
    score = torch.full((s.B, s.L), float("inf"), device="cuda")
    argmax = torch.full((s.B, s.L), -1, dtype=torch.int32, device="cuda")
    margin = torch.full((s.B, s.L), -1.0, device="cuda")
    dl.dllm_confidence(logits, R_max=s.Lw, count=count, out_idx=idx, out_cols=s.L,
                       conf_out=score, argmax_out=argmax, margin_out=margin, dev_status=st)
    start = torch.full((s.B,), w, dtype=torch.int32, device="cuda")
    length = dl.dllm_stable_prefix(score, start, 0.9, min_commit=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0

    ref_cos = oracle.saliency_cos(f64(inp["cur"][:, w:]), f64(inp["prev"][:, w:]))
    assert np.max(np.abs(f64(cos) - ref_cos)) <= SCORE_TOL
    ref_idx, ref_count = oracle.compact(oracle.salient_flags(i32(cos), s.tau, None), w)
    assert np.array_equal(i32(count), ref_count) and np.array_equal(i32(idx), ref_idx)
    assert ref_count.tolist() == [n_act] * s.B
    for b in range(s.B):  # the planted positions are the selected ones
        assert np.array_equal(ref_idx[b, :n_act], inp["planted"][b].numpy())
    kc_ref, vc_ref = oracle.kv_scatter(f64(inp["k_cache"]), f64(inp["v_cache"]), f64(inp["k_new"]),
                                       f64(inp["v_new"]), ref_idx, ref_count)
    assert np.array_equal(f64(t["k_cache"]), kc_ref) and np.array_equal(f64(t["v_cache"]), vc_ref)
    _check_attention_heads(o, lse, cs, f64(inp["q"]), kc_ref, vc_ref, [n_act] * s.B,
                           [(0, 0), (1, 9), (2, 20), (3, 31)])
    # confidence of every active row, read back at its position
    rc, ra, rm = oracle.confidence(f64(logits_rows), count=[n_act] * s.B)
    gsc, gam, gmg = f64(score), i32(argmax), f64(margin)
    for b in range(s.B):
        pos = ref_idx[b, :n_act]
        assert np.all(np.abs(gsc[b, pos] - rc[b, :n_act]) <= 1e-6 + SCORE_TOL * np.abs(rc[b, :n_act]))
        assert np.array_equal(gam[b, pos], ra[b, :n_act])
        assert np.max(np.abs(gmg[b, pos] - rm[b, :n_act])) <= 1e-6
    assert np.array_equal(i32(length), oracle.stable_prefix(gsc.astype(np.float32), [w] * s.B,
                                                            0.9, True))
