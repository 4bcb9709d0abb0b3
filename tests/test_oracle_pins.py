"""Pins of the float64 oracle to things other than itself.

Each test ties one oracle output to a closed form, a hand-derived fixture
(``tests/golden/closed_forms.json``), a library routine evaluating the same
mathematics by another route, brute force on tiny inputs, or an invariant that
characterises the output uniquely.  None of them needs a GPU.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- cosine

def test_cos_golden(golden):
    for case in golden["cosine"]:
        c = oracle.saliency_cos(np.array([case["cur"]]), np.array([case["prev"]]))[0]
        assert abs(c - case["cos"]) < 1e-15, case


def test_cos_identity_negation_scale():
    x = RNG.standard_normal((5, 7, 33))
    assert np.allclose(oracle.saliency_cos(x, x), 1.0, atol=1e-15, rtol=0)
    assert np.allclose(oracle.saliency_cos(x, -x), -1.0, atol=1e-15, rtol=0)
    assert np.allclose(oracle.saliency_cos(x, 3.5 * x), 1.0, atol=1e-15, rtol=0)
    y = RNG.standard_normal((5, 7, 33))
    assert np.allclose(oracle.saliency_cos(2.0 * x, 0.25 * y), oracle.saliency_cos(x, y), atol=1e-14)
    # symmetric in its arguments
    assert np.allclose(oracle.saliency_cos(x, y), oracle.saliency_cos(y, x), atol=1e-15)


def test_cos_orthogonal():
    x = RNG.standard_normal((64, 40))
    y = RNG.standard_normal((64, 40))
    y -= (np.sum(x * y, -1) / np.sum(x * x, -1))[:, None] * x  # Gram-Schmidt
    assert np.allclose(oracle.saliency_cos(x, y), 0.0, atol=1e-13)


def test_cos_matches_torch_library():
    x = RNG.standard_normal((3, 50, 128))
    y = x + 0.3 * RNG.standard_normal((3, 50, 128))
    ref = torch.nn.functional.cosine_similarity(torch.from_numpy(x), torch.from_numpy(y), dim=-1)
    assert np.allclose(oracle.saliency_cos(x, y), ref.numpy(), atol=1e-14, rtol=0)


def test_cos_zero_norm_readings():
    z = np.zeros((1, 2, 4))
    a = np.ones((1, 2, 4))
    assert np.all(oracle.saliency_cos(z, z) == 1.0)
    assert np.all(oracle.saliency_cos(z, a) == 0.0)
    assert np.all(oracle.saliency_cos(a, z) == 0.0)


def test_cos_value_on_planted_rows():
    # cur = prev + N(0, 0.5) gives cos -> 1/sqrt(1.25) for large D; N(0, 1e-3) gives ~1 - 5e-7.
    g = torch.Generator().manual_seed(7)
    prev = torch.randn((200, 4096), generator=g, dtype=torch.float64)
    big = prev + 0.5 * torch.randn((200, 4096), generator=g, dtype=torch.float64)
    small = prev + 1e-3 * torch.randn((200, 4096), generator=g, dtype=torch.float64)
    assert abs(oracle.saliency_cos(big, prev).mean() - 1 / math.sqrt(1.25)) < 2e-3
    assert abs(oracle.saliency_cos(small, prev).mean() - (1 - 5e-7)) < 1e-7


# ---------------------------------------------------------------- flags / compaction

def test_flags_threshold_edges():
    cos = np.array([[0.5, 0.99, 0.98999, np.nan, 1.0]], dtype=np.float32)
    f = oracle.salient_flags(cos, 0.99)
    assert f.tolist() == [[True, False, True, True, False]]
    assert oracle.salient_flags(cos, 2.0).all()
    assert oracle.salient_flags(cos, -2.0).tolist() == [[False, False, False, True, False]]
    locked = np.array([[1, 0, 0, 1, 0]], dtype=np.uint8)
    assert oracle.salient_flags(cos, 2.0, locked).tolist() == [[False, True, True, False, True]]


@pytest.mark.parametrize("n", [1, 2, 5, 10])
def test_compaction_brute_force(n):
    # The invariants below (length = popcount, strictly increasing, each entry
    # flagged, -1 padding) characterise the ordered compaction uniquely.
    for bits in itertools.product([False, True], repeat=n):
        flags = np.array([bits, bits[::-1]])
        for base in (0, 7):
            idx, count = oracle.compact(flags, base)
            for b in range(2):
                c = int(count[b])
                assert c == int(flags[b].sum())
                sel = idx[b, :c] - base
                assert np.all(np.diff(sel) > 0)
                assert np.all(flags[b][sel])
                assert np.all(idx[b, c:] == -1)


def test_select_recovers_planted_set_tiny():
    s = workloads.TINY_F32
    inp = workloads.make_step(s)
    cos, idx, count = oracle.saliency_select(inp["cur"].double().numpy(),
                                             inp["prev"].double().numpy(), s.tau)
    assert int(count[0]) == s.n_salient
    assert idx[0, : count[0]].tolist() == inp["planted"][0].tolist()


def test_select_recovers_planted_set_1k_window():
    s = workloads.STEP_1K
    inp = workloads.make_step(s, with_logits=False)
    w = s.win_start
    cos, idx, count = oracle.saliency_select(inp["cur"][:, w:].double().numpy(),
                                             inp["prev"][:, w:].double().numpy(), s.tau,
                                             idx_base=w)
    assert int(count[0]) == s.n_salient
    assert idx[0, : count[0]].tolist() == inp["planted"][0].tolist()
    assert cos[0].min() > 0.85 and cos[0].max() <= 1.0 + 1e-12


def test_select_with_cluster_pattern_and_locks():
    s = workloads.TINY_F32
    inp = workloads.make_step(s, pattern="cluster", n_salient=40)
    cur, prev = inp["cur"].double().numpy(), inp["prev"].double().numpy()
    planted = inp["planted"][0].tolist()
    locked = np.zeros((1, s.L), dtype=np.uint8)
    locked[0, planted[:5]] = 1
    _, idx, count = oracle.saliency_select(cur, prev, s.tau, locked)
    assert idx[0, : count[0]].tolist() == planted[5:]


# ---------------------------------------------------------------- confidence

def test_confidence_golden(golden):
    for case in golden["confidence"]:
        conf, am, mg = oracle.confidence(np.array([[case["logits"]]]))
        assert abs(conf[0, 0] - case["conf"]) < 1e-15
        assert am[0, 0] == case["argmax"]
        assert mg[0, 0] == case["margin"]


@pytest.mark.parametrize("V", [2, 3, 17, 1000])
@pytest.mark.parametrize("c", [0.5, 4.0, -3.0])
def test_confidence_one_hot_closed_form(V, c):
    z = np.zeros((1, 1, V))
    z[0, 0, 0] = c
    conf, am, mg = oracle.confidence(z)
    if c > 0:
        assert abs(conf[0, 0] - math.exp(c) / (math.exp(c) + V - 1)) < 1e-15
        assert am[0, 0] == 0 and abs(mg[0, 0] - c) < 1e-15
    else:  # the maximum 0 is first reached at index 1 (index 0 holds c < 0)
        assert am[0, 0] == 1
        if V > 2:
            assert mg[0, 0] == 0.0
        assert abs(conf[0, 0] - 1.0 / (math.exp(c) + V - 1)) < 1e-15


def test_confidence_uniform():
    conf, am, mg = oracle.confidence(np.full((1, 3, 50), 1.7))
    assert np.allclose(conf, 1 / 50, atol=1e-16, rtol=0)
    assert np.all(am == 0) and np.all(mg == 0)


def test_confidence_matches_torch_library():
    z = 2.0 * RNG.standard_normal((2, 6, 3001))
    conf, am, mg = oracle.confidence(z)
    t = torch.from_numpy(z)
    p = torch.softmax(t, dim=-1)
    assert np.allclose(conf, p.max(-1).values.numpy(), atol=1e-15, rtol=1e-12)
    assert np.array_equal(am, torch.argmax(t, -1).numpy())
    top2 = torch.topk(t, 2, dim=-1).values
    assert np.allclose(mg, (top2[..., 0] - top2[..., 1]).numpy(), atol=0, rtol=0)


def test_confidence_shift_invariance():
    z = RNG.standard_normal((1, 4, 300))
    a = oracle.confidence(z)
    b = oracle.confidence(z + 123.25)
    assert np.allclose(a[0], b[0], atol=1e-14)
    assert np.array_equal(a[1], b[1])
    assert np.allclose(a[2], b[2], atol=1e-12)


def test_confidence_brute_force_small_V():
    for V in range(2, 9):
        z = np.round(RNG.standard_normal((1, 5, V)) * 2, 1)  # rounding makes ties likely
        conf, am, mg = oracle.confidence(z)
        for r in range(5):
            row = [float(x) for x in z[0, r]]
            best = 0
            for j in range(1, V):
                if row[j] > row[best]:
                    best = j
            total = 0.0
            for j in range(V):
                total += math.exp(row[j] - row[best])
            second = max(row[j] for j in range(V) if j != best)
            assert am[0, r] == best
            assert abs(conf[0, r] - 1.0 / total) < 1e-15
            assert mg[0, r] == row[best] - second


def test_confidence_row_idx_and_count():
    z = RNG.standard_normal((2, 10, 20))
    row_idx = np.array([[3, 1, 9, 0], [2, 2, 5, 7]], dtype=np.int32)
    count = np.array([3, 1])
    conf, am, mg = oracle.confidence(z, count=count, row_idx=row_idx)
    full_conf, full_am, _ = oracle.confidence(z)
    for b in range(2):
        for r in range(4):
            if r < count[b]:
                assert conf[b, r] == full_conf[b, row_idx[b, r]]
                assert am[b, r] == full_am[b, row_idx[b, r]]
            else:
                assert np.isnan(conf[b, r]) and am[b, r] == -1


# ---------------------------------------------------------------- scatter

def test_scatter_properties():
    B, L, H, d, M = 2, 40, 3, 8, 12
    kc = RNG.standard_normal((B, L, H, d))
    vc = RNG.standard_normal((B, L, H, d))
    kn = RNG.standard_normal((B, M, H, d))
    vn = RNG.standard_normal((B, M, H, d))
    idx = np.full((B, M), -1, dtype=np.int32)
    idx[0, :5] = [0, 3, 4, 5, 39]
    idx[1, :0] = []
    count = np.array([5, 0])
    k2, v2 = oracle.kv_scatter(kc, vc, kn, vn, idx, count)
    assert np.array_equal(k2[0, idx[0, :5]], kn[0, :5])
    assert np.array_equal(v2[0, idx[0, :5]], vn[0, :5])
    untouched = np.setdiff1d(np.arange(L), idx[0, :5])
    assert np.array_equal(k2[0, untouched], kc[0, untouched])
    assert np.array_equal(k2[1], kc[1]) and np.array_equal(v2[1], vc[1])
    assert not np.shares_memory(k2, kc)


# ---------------------------------------------------------------- attention

def test_attention_golden(golden):
    for case in golden["attention"]:
        q = np.array(case["q"])[None, :, None, :]
        k = np.array(case["k"])[None, :, None, :]
        v = np.array(case["v"])[None, :, None, :]
        o, lse, cs = oracle.partial_attention(q, k, v, [1])
        assert np.allclose(o[0, 0, 0], case["o"], atol=1e-14, rtol=0)
        assert abs(lse[0, 0, 0] - case["lse"]) < 1e-14
        assert np.allclose(cs[0, 0], case["colsum"], atol=1e-15, rtol=0)


def _rand_attn(B, M, L, H, d, seed=0):
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, M, H, d)), r.standard_normal((B, L, H, d)),
            r.standard_normal((B, L, H, d)))


def test_attention_all_active_equals_torch_sdpa():
    B, L, H, d = 2, 37, 3, 16
    q, k, v = _rand_attn(B, L, L, H, d)
    o, lse, cs = oracle.partial_attention(q, k, v, [L, L])
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k).permute(0, 2, 1, 3)
    tv = torch.from_numpy(v).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv).permute(0, 2, 1, 3)
    assert np.allclose(o, ref.numpy(), atol=1e-12, rtol=0)
    s = torch.matmul(tq, tk.transpose(-1, -2)) / math.sqrt(d)
    assert np.allclose(lse, torch.logsumexp(s, -1).numpy(), atol=1e-12, rtol=0)
    # full-matrix column sums when every row is active
    assert np.allclose(cs, torch.softmax(s, -1).sum(-2).numpy(), atol=1e-12, rtol=0)


def test_attention_zero_query_gives_mean_and_uniform_colsum():
    B, M, L, H, d = 1, 9, 23, 2, 8
    q, k, v = _rand_attn(B, M, L, H, d, 3)
    q[:] = 0
    o, lse, cs = oracle.partial_attention(q, k, v, [7])
    assert np.allclose(o[0, :7], np.broadcast_to(v[0].mean(0), (7, H, d)), atol=1e-14)
    assert np.allclose(lse[0, :, :7], math.log(L), atol=1e-14)
    assert np.allclose(cs, 7 / L, atol=1e-14, rtol=0)
    assert np.all(np.isnan(o[0, 7:]))


def test_attention_single_key():
    q, k, v = _rand_attn(1, 4, 1, 2, 8, 5)
    o, lse, cs = oracle.partial_attention(q, k, v, [4])
    assert np.allclose(o[0], np.broadcast_to(v[0, 0], (4, 2, 8)), atol=1e-15)
    s = np.einsum("mhd,hd->hm", q[0], k[0, 0]) / math.sqrt(8)
    assert np.allclose(lse[0], s, atol=1e-14)
    assert np.allclose(cs, 4.0, atol=1e-14)


def test_attention_key_permutation_invariance():
    q, k, v = _rand_attn(1, 6, 31, 2, 16, 9)
    perm = RNG.permutation(31)
    a = oracle.partial_attention(q, k, v, [6])
    b = oracle.partial_attention(q, k[:, perm], v[:, perm], [6])
    assert np.allclose(a[0], b[0], atol=1e-14)
    assert np.allclose(a[1], b[1], atol=1e-14)
    assert np.allclose(a[2][..., perm], b[2], atol=1e-15)


def test_attention_brute_force_tiny():
    for L in range(1, 9):
        q, k, v = _rand_attn(1, 3, L, 2, 4, L)
        scale = 0.37
        o, lse, cs = oracle.partial_attention(q, k, v, [2], scale)
        for h in range(2):
            col = [0.0] * L
            for i in range(2):
                s = [scale * sum(q[0, i, h, t] * k[0, j, h, t] for t in range(4)) for j in range(L)]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                tot = sum(w)
                for t in range(4):
                    ref = sum(w[j] * v[0, j, h, t] for j in range(L)) / tot
                    assert abs(o[0, i, h, t] - ref) < 1e-13
                assert abs(lse[0, h, i] - (mx + math.log(tot))) < 1e-13
                for j in range(L):
                    col[j] += w[j] / tot
            assert np.allclose(cs[0, h], col, atol=1e-14, rtol=0)


def test_attention_colsum_sums_to_count_and_ignores_padding():
    q, k, v = _rand_attn(2, 20, 45, 3, 8, 11)
    a = oracle.partial_attention(q, k, v, [13, 0])
    assert np.allclose(a[2][0].sum(-1), 13, atol=1e-12)
    assert np.all(a[2][1] == 0)
    q2 = q.copy()
    q2[0, 13:] = 1e3  # garbage in padded rows must not matter
    b = oracle.partial_attention(q2, k, v, [13, 0])
    assert np.array_equal(a[0][0, :13], b[0][0, :13])
    assert np.array_equal(a[2], b[2])


# ---------------------------------------------------------------- stable prefix

def test_prefix_golden(golden):
    for case in golden["stable_prefix"]:
        score = np.array([case["score"]], dtype=np.float32)
        for c in case["cases"]:
            got = oracle.stable_prefix(score, [c["start"]], case["tau"], c["min_commit"])
            assert got[0] == c["len"], c


@pytest.mark.parametrize("n", [1, 3, 6, 10])
def test_prefix_brute_force(n):
    # len is characterised by: every position in [start, start+len) stable and
    # (start+len == L or position start+len unstable), then the fallback.
    for bits in itertools.product([False, True], repeat=n):
        score = np.where(np.array(bits), 0.95, 0.2).astype(np.float32)[None, :]
        for start in range(n + 1):
            for mc in (False, True):
                got = int(oracle.stable_prefix(score, [start], 0.9, mc)[0])
                k = got
                if mc and start < n and not bits[start]:
                    assert k == 1
                    continue
                assert all(bits[start:start + k])
                assert start + k == n or not bits[start + k]


def test_prefix_nan_and_equality():
    s = np.array([[0.9, np.nan, 1.0], [np.inf, np.inf, 0.9]], dtype=np.float32)
    got = oracle.stable_prefix(s, [0, 0], 0.9, False)
    assert got.tolist() == [1, 3]


# ---------------------------------------------------------------- whole step

def _tiny_step_inputs():
    s = workloads.TINY_F32
    inp = workloads.make_step(s)
    d = {k: inp[k].double().numpy() for k in ("cur", "prev", "k_cache", "v_cache",
                                               "k_new", "v_new", "q", "logits")}
    return s, inp, d


def test_step_all_salient_is_dense_step():
    s, inp, d = _tiny_step_inputs()
    score = np.full((1, s.L), np.inf)
    out = oracle.step(d["cur"], d["prev"], d["k_cache"], d["v_cache"], d["k_new"],
                      d["v_new"], d["q"], d["logits"], tau=2.0, win_start=0,
                      score=score, start=[0], tau_c=0.9)
    assert int(out["count"][0]) == s.L
    # every cache row replaced, and attention is dense attention over the new cache
    assert np.array_equal(out["k_cache"], d["k_new"])
    tq = torch.from_numpy(d["q"]).permute(0, 2, 1, 3)
    tk = torch.from_numpy(d["k_new"]).permute(0, 2, 1, 3)
    tv = torch.from_numpy(d["v_new"]).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv).permute(0, 2, 1, 3)
    assert np.allclose(out["o"], ref.numpy(), atol=1e-13)


def test_step_nothing_salient():
    s, inp, d = _tiny_step_inputs()
    score = np.full((1, s.L), np.inf)
    out = oracle.step(d["cur"], d["prev"], d["k_cache"], d["v_cache"], d["k_new"],
                      d["v_new"], d["q"], d["logits"], tau=-2.0, win_start=0,
                      score=score, start=[0], tau_c=0.9)
    assert int(out["count"][0]) == 0
    assert np.array_equal(out["k_cache"], d["k_cache"])
    assert np.all(out["colsum"] == 0)
    assert np.all(np.isnan(out["o"]))


# ---------------------------------------------------------------- lock criterion

def test_lock_kl_golden(golden):
    for case in golden["lock_kl"]:
        kl, unc = oracle.lock_kl(np.array([[case["cur"]]]), np.array([[case["prev"]]]))
        assert abs(kl[0, 0] - case["kl"]) < 1e-14, case
        assert abs(unc[0, 0] - case["unc"]) < 1e-14, case


def test_lock_kl_matches_scipy_entropy():
    from scipy.special import softmax
    from scipy.stats import entropy
    z = RNG.standard_normal((2, 5, 300)) * 2.0
    y = z + RNG.standard_normal((2, 5, 300)) * 0.3
    kl, unc = oracle.lock_kl(z, y)
    for b in range(2):
        for r in range(5):
            p, q = softmax(z[b, r]), softmax(y[b, r])
            assert abs(kl[b, r] - entropy(p, q)) < 1e-12
            assert abs(unc[b, r] - (1.0 - p.max())) < 1e-14


def test_lock_kl_identity_shift_and_gibbs():
    z = RNG.standard_normal((1, 6, 50))
    kl, _ = oracle.lock_kl(z, z + 7.5)  # same distribution
    assert np.max(np.abs(kl)) < 1e-13
    y = RNG.standard_normal((1, 6, 50))
    kl, _ = oracle.lock_kl(z, y)
    assert np.all(kl > 0)


def test_lock_kl_brute_force_small_vocab():
    for V in (2, 3, 4):
        z = RNG.standard_normal((1, 3, V)) * 3
        y = RNG.standard_normal((1, 3, V)) * 3
        kl, unc = oracle.lock_kl(z, y)
        for r in range(3):
            ez = [math.exp(v) for v in z[0, r]]
            ey = [math.exp(v) for v in y[0, r]]
            p = [e / sum(ez) for e in ez]
            q = [e / sum(ey) for e in ey]
            ref = sum(pj * math.log(pj / qj) for pj, qj in zip(p, q))
            assert abs(kl[0, r] - ref) < 1e-12
            assert abs(unc[0, r] - (1 - max(p))) < 1e-14


def test_lock_kl_row_idx_and_count():
    z = RNG.standard_normal((2, 6, 40))
    y = RNG.standard_normal((2, 6, 40))
    row_idx = np.array([[5, 0, 3], [1, 1, 2]])
    kl, unc = oracle.lock_kl(z, y, count=[3, 1], row_idx=row_idx)
    full, ufull = oracle.lock_kl(z, y)
    assert np.allclose(kl[0], full[0, [5, 0, 3]], rtol=0, atol=0)
    assert kl[1, 0] == full[1, 1] and np.all(np.isnan(kl[1, 1:]))


def test_lock_decision_without_gate_and_with_numpy_quantile():
    kl = RNG.random((3, 40)).astype(np.float32) * 1e-2
    unc = RNG.random((3, 40)).astype(np.float32)
    count = [40, 17, 0]
    lock = oracle.lock_decision(kl, unc, count, 5e-3, 0.0)
    for b, n in enumerate(count):
        assert np.array_equal(lock[b, :n], kl[b, :n] < np.float32(5e-3))
        assert not lock[b, n:].any()
    for q in (0.1, 0.25, 0.5, 0.9):
        lock = oracle.lock_decision(kl, unc, count, 5e-3, q)
        for b, n in enumerate(count[:2]):
            t = np.quantile(unc[b, :n], q, method="inverted_cdf")
            assert np.array_equal(lock[b, :n], (kl[b, :n] < np.float32(5e-3)) & (unc[b, :n] <= t))


def test_lock_decision_gate_extremes_and_nan():
    kl = np.zeros((1, 8), dtype=np.float32)
    unc = np.array([[0.5, 0.1, 0.3, 0.1, 0.9, 0.2, 0.7, 0.4]], dtype=np.float32)
    lock = oracle.lock_decision(kl, unc, [8], 1.0, 1.0 / 8)
    assert lock[0].tolist() == [False, True, False, True, False, False, False, False]  # tie at the minimum
    assert oracle.lock_decision(kl, unc, [8], 1.0, 1.0).all()  # q >= 1: no gate
    kl[0, 2] = np.nan
    assert not oracle.lock_decision(kl, unc, [8], 1.0, 0.0)[0, 2]


# ---------------------------------------------------------------- adaptive prefix

def test_adaptive_prefix_golden(golden):
    for case in golden["adaptive_prefix"]:
        ln, tau = oracle.adaptive_prefix(np.array([case["score"]]), [case["start"]], case["lo"],
                                         case["hi"])
        assert ln[0] == case["len"], case
        assert tau[0] == np.float32(case["tau"]), case


def test_adaptive_prefix_brute_force_characterisation():
    # For every pattern: tau is the minimum of the first k_lo active scores
    # (numpy), every committed score is >= tau, and len is the largest k <=
    # k_hi with that property, at least 1.
    vals = np.array([0.2, 0.5, 0.8], dtype=np.float32)
    for n in (1, 2, 3, 5, 6):
        for pat in itertools.product(range(3), repeat=n):
            score = vals[list(pat)][None, :]
            for start in range(n + 1):
                for lo, hi in ((0.25, 0.5), (0.1, 0.9), (0.5, 0.5)):
                    ln, tau = oracle.adaptive_prefix(score, [start], lo, hi)
                    A = n - start
                    if A == 0:
                        assert ln[0] == 0 and np.isinf(tau[0])
                        continue
                    k_lo = min(A, max(1, math.ceil(float(np.float32(lo)) * A)))
                    k_hi = max(k_lo, math.floor(float(np.float32(hi)) * A))
                    seg = score[0, start:]
                    assert tau[0] == np.min(seg[:k_lo])
                    feasible = [k for k in range(1, k_hi + 1) if np.all(seg[:k] >= tau[0])]
                    assert ln[0] == max(feasible + [1])
                    assert np.array_equal(np.minimum.accumulate(seg)[:ln[0]] >= tau[0],
                                          np.ones(ln[0], dtype=bool))


def test_adaptive_prefix_nan_stops_and_fallback():
    score = np.array([[0.9, np.nan, 0.9, 0.9], [np.nan, 0.9, 0.9, 0.9]], dtype=np.float32)
    ln, tau = oracle.adaptive_prefix(score, [0, 0], 0.25, 1.0)
    assert ln.tolist() == [1, 1]


# ---------------------------------------------------------------- approximate attention update

def _attention_all_rows(q, k, v, scale=None):
    B, L = q.shape[:2]
    return oracle.partial_attention(q, k, v, [L] * B, scale=scale)


def test_approx_update_golden(golden):
    for case in golden["approx_attention"]:
        q = np.array(case["q"])[None, None, None, :]           # [1, 1, 1, d]
        k = np.array(case["k"])[None, :, None, :]              # [1, 2, 1, d]
        v = np.array(case["v_prev"])[None, :, None, :]
        o_prev, lse, _ = oracle.partial_attention(q, k, v, [1], scale=case["scale"])
        # the query row is position 0; position 1 is salient
        L = k.shape[1]
        qa = np.zeros((1, L, 1, q.shape[-1])); qa[:, 0] = q[:, 0]
        oa = np.zeros((1, L, 1, q.shape[-1])); oa[:, 0] = o_prev[:, 0]
        la = np.zeros((1, 1, L)); la[:, :, 0] = lse[:, :, 0]
        v_new = np.array(case["v_new_pos1"])[None, None, None, :]
        o = oracle.approx_attention_update(oa, qa, la, k, v, v_new, [[1]], [1], [[0]], [1],
                                           scale=case["scale"])
        assert np.allclose(o[0, 0, 0], case["o_new"], atol=1e-14, rtol=0), (o[0, 0, 0], case)


@pytest.mark.parametrize("scale", [None, 0.3])
def test_approx_update_exact_when_only_values_change(scale):
    """With queries and keys unchanged the attention weights do not change,
    so the update of the non-salient path is exact: it must equal attention
    recomputed over the updated value cache, for every stable row."""
    B, L, H, d = 2, 13, 3, 8
    q = RNG.standard_normal((B, L, H, d))
    k = RNG.standard_normal((B, L, H, d))
    v = RNG.standard_normal((B, L, H, d))
    o_prev, lse, _ = _attention_all_rows(q, k, v, scale)
    counts = [4, 1]
    idx = np.full((B, L), -1)
    idx[0, :4] = [1, 5, 6, 12]
    idx[1, :1] = [0]
    v_new = RNG.standard_normal((B, L, H, d))
    stable = np.full((B, L), -1)
    s_counts = []
    for b in range(B):
        rest = [j for j in range(L) if j not in set(idx[b, :counts[b]])]
        stable[b, :len(rest)] = rest
        s_counts.append(len(rest))
    o = oracle.approx_attention_update(o_prev, q, lse, k, v, v_new, idx, counts, stable, s_counts,
                                       scale=scale)
    _, v_upd = oracle.kv_scatter(k, v, k, v_new, idx, counts)
    o_exact, _, _ = _attention_all_rows(q, k, v_upd, scale)
    for b in range(B):
        rows = stable[b, :s_counts[b]]
        assert np.max(np.abs(o[b, rows] - o_exact[b, rows])) < 1e-12
        sal = idx[b, :counts[b]]
        assert np.array_equal(o[b, sal], o_prev[b, sal])  # only stable rows change


def test_approx_update_no_change_cases():
    B, L, H, d = 1, 9, 2, 4
    q, k, v = (RNG.standard_normal((B, L, H, d)) for _ in range(3))
    o_prev, lse, _ = _attention_all_rows(q, k, v)
    idx = np.array([[2, 7] + [-1] * 7])
    stable = np.array([[0, 1, 3, 4, 5, 6, 8, -1, -1]])
    v_same = np.zeros((B, L, H, d))
    v_same[0, :2] = v[0, [2, 7]]
    o = oracle.approx_attention_update(o_prev, q, lse, k, v, v_same, idx, [2], stable, [7])
    assert np.max(np.abs(o - o_prev)) < 1e-15                       # dV = 0
    o = oracle.approx_attention_update(o_prev, q, lse, k, v, v_same + 1, idx, [0], stable, [7])
    assert np.array_equal(o, o_prev)                                 # no salient token
    o = oracle.approx_attention_update(o_prev, q, lse, k, v, v_same + 1, idx, [2], stable, [0])
    assert np.array_equal(o, o_prev)                                 # no stable row


# ---------------------------------------------------------------- Attn-Sampler order

def test_attn_sampler_golden(golden):
    for case in golden["attn_sampler"]:
        order, n = oracle.attn_sampler_select(np.array([case["score"]]),
                                              np.array([case["candidates"]]), case["tau"],
                                              case["gamma"], case["k_max"])
        assert order[0].tolist() == case["order"] and int(n[0]) == case["n"], case


def test_attn_scores_sum_heads_and_layers():
    # the row-softmax probabilities of each active row add up to 1 per head,
    # so the scores of a batch row add up to H * count
    B, L, H, d = 2, 11, 3, 8
    q, k, v = (RNG.standard_normal((B, L, H, d)) for _ in range(3))
    _, _, colsum = oracle.partial_attention(q, k, v, [5, 11])
    a = oracle.attn_scores(colsum)
    assert a.shape == (B, L)
    assert np.allclose(a.sum(axis=1), [H * 5, H * 11], atol=1e-12, rtol=0)
    per_layer = np.stack([colsum, 2 * colsum], axis=1)           # [B, layers, H, L]
    assert np.allclose(oracle.attn_scores(per_layer), 3 * a, atol=1e-12, rtol=0)


def test_attn_sampler_order_matches_lexsort():
    B, L = 4, 200
    score = np.round(RNG.standard_normal((B, L)) * 4) / 4          # many ties
    cand = RNG.random((B, L)) < 0.7
    order, n = oracle.attn_sampler_select(score, cand, -np.inf, 0.0, 0)
    for b in range(B):
        pos = np.nonzero(cand[b])[0]
        ref = pos[np.lexsort((pos, -score[b, pos].astype(np.float32)))]
        assert np.array_equal(order[b, :len(pos)], ref)
        assert np.all(order[b, len(pos):] == -1)
        assert n[b] == len(pos)                                     # threshold -inf: all


def test_attn_sampler_count_brute_force():
    """n is the largest k <= cap such that the k leading entries reach the
    threshold (at least 1); checked over all threshold, fraction and cap
    settings of small random cases."""
    for trial in range(200):
        L = 1 + trial % 9
        score = np.round(RNG.random((1, L)) * 8) / 8
        cand = RNG.random((1, L)) < 0.8
        for tau, gamma, k_max in itertools.product([0.0, 0.3, 0.9], [0.0, 0.5, 1.0], [0, 1, 3]):
            order, n = oracle.attn_sampler_select(score, cand, tau, gamma, k_max)
            o = [j for j in order[0] if j >= 0]
            if not o:
                assert n[0] == 0
                continue
            thr = np.float32(tau)
            if gamma > 0:
                thr = max(thr, np.float32(gamma) * np.float32(score[0, o[0]]))
            best = 0
            for kk in range(1, len(o) + 1):
                if all(np.float32(score[0, j]) >= thr for j in o[:kk]) and (k_max <= 0 or kk <= k_max):
                    best = kk
            assert n[0] == max(best, 1)


def test_attn_sampler_nan_and_signed_zero():
    score = np.array([[np.nan, 0.0, -0.0, 1.0, -np.inf]])
    order, n = oracle.attn_sampler_select(score, None, -1.0, 0.0, 0)
    # 1.0, then the two zeros by position (-0 == +0), -inf, NaN last
    assert order[0].tolist() == [3, 1, 2, 4, 0]
    assert n[0] == 3


# ---------------------------------------------------------------- SlowFast phases

def test_slowfast_golden(golden):
    for case in golden["slowfast"]:
        starts = [[s] for s in case["start"]]
        preds = [[e] for e in case["e_cand"]]
        phase, end = oracle.slowfast_phases(starts, preds, case["window"], case["sigma2"])
        assert phase[:, 0].tolist() == case["phase"], case
        assert end[:, 0].tolist() == case["region_end"], case


def test_slowfast_matches_numpy_variance():
    """Away from exact ties the integer form is numpy's population variance
    of the window below sigma2; a cycle restarts after each fast step."""
    for trial in range(40):
        W = 1 + trial % 5
        sigma2 = [0.3, 1.7, 4.9, 0.0][trial % 4] + 1e-7  # never a multiple of 1 / W^2
        T = 60
        e = np.cumsum(RNG.integers(0, 3, T)) + RNG.integers(0, 2, T)
        starts = np.minimum(e - RNG.integers(0, 4, T), e).astype(int)
        phase, end = oracle.slowfast_phases(starts[:, None], e[:, None], W, sigma2)
        hist = []
        for t in range(T):
            hist = (hist + [int(e[t])])[-W:]
            fast = len(hist) == W and hist[-1] > starts[t] and np.var(hist) < sigma2
            assert phase[t, 0] == int(fast) and end[t, 0] == (hist[-1] if fast else -1)
            if fast:
                hist = []


def test_slowfast_special_cases():
    # a prediction that never moves past the start never decodes fast
    ph, _ = oracle.slowfast_phases([[5]] * 10, [[5]] * 10, 3, 100.0)
    assert ph.sum() == 0
    # sigma2 = 0: the variance is never below it
    ph, _ = oracle.slowfast_phases([[0]] * 10, [[7]] * 10, 2, 0.0)
    assert ph.sum() == 0
    # a constant prediction beyond the start: fast every W steps
    ph, end = oracle.slowfast_phases([[0]] * 12, [[7]] * 12, 3, 0.1)
    assert ph[:, 0].tolist() == [0, 0, 1] * 4 and set(end[ph[:, 0] == 1, 0]) == {7}
    # window 1: fast whenever the prediction lies beyond the start
    ph, _ = oracle.slowfast_phases([[0], [3], [3]], [[2], [3], [9]], 1, 0.5)
    assert ph[:, 0].tolist() == [1, 0, 1]


# ---------------------------------------------------------------- structural snapping

def test_snap_prefix_golden(golden):
    for case in golden["snap_prefix"]:
        V = 1 + max(max(case["tokens"]), max(case["delim_ids"]))
        delim = np.zeros(V, dtype=np.uint8)
        delim[case["delim_ids"]] = 1
        got = oracle.snap_prefix(np.array([case["tokens"]]), delim, [case["start"]],
                                 [case["length"]], case["min_len"])
        assert int(got[0]) == case["snapped"], case


def test_snap_prefix_characterisation():
    """The snapped block ends on a delimiter at or after the minimum and no
    delimiter lies between its end and the original end; without such a
    delimiter the length is unchanged; it never grows."""
    for trial in range(300):
        L, V = 1 + trial % 23, 6
        tok = RNG.integers(0, V, (1, L))
        delim = (RNG.random(V) < 0.3).astype(np.uint8)
        s = int(RNG.integers(0, L))
        n = int(RNG.integers(0, L - s + 1))
        m = int(RNG.integers(0, n + 2))
        got = int(oracle.snap_prefix(tok, delim, [s], [n], m)[0])
        lo = s + max(m, 1) - 1
        ends = [p for p in range(lo, s + n) if delim[tok[0, p]]]
        if ends:
            assert got == max(ends) - s + 1 and delim[tok[0, s + got - 1]]
        else:
            assert got == n
        assert got <= n


# ---------------------------------------------------------------- SlowFast token selection

def test_slowfast_select_golden(golden):
    for case in golden["slowfast_select"]:
        conf = np.array([case["conf"]], dtype=np.float64)
        masked = np.array([case["masked"]], dtype=np.uint8)
        idx, count = oracle.slowfast_select(conf, masked, [case["start"]], [case["phase"]],
                                            [case["region_end"]], case["tau_high"],
                                            case["width"], case["k"])
        n = len(case["idx"])
        assert count.tolist() == [n], case["derivation"]
        assert idx[0, :n].tolist() == case["idx"], case["derivation"]
        assert np.all(idx[0, n:] == -1)


def test_slowfast_slow_select_matches_lexsort():
    """The slow phase's top k against numpy's lexsort ranking (descending
    float32 confidence, then ascending position) of the window's masked,
    non-NaN candidates, with ties and NaN in the draws."""
    rng = np.random.default_rng(5)
    B, L = 6, 300
    conf = np.round(rng.random((B, L)), 2)  # two decimals: many ties
    conf[rng.random((B, L)) < 0.05] = np.nan
    masked = (rng.random((B, L)) < 0.7).astype(np.uint8)
    for width, k in ((50, 1), (64, 7), (300, 40), (17, 100)):
        start = rng.integers(0, L, B)
        idx, count = oracle.slowfast_slow_select(conf, masked, start, width, k)
        for b in range(B):
            lo, hi = start[b], min(start[b] + width, L)
            pos = np.arange(lo, hi)
            c32 = conf[b, lo:hi].astype(np.float32)
            keep = (masked[b, lo:hi] != 0) & ~np.isnan(c32)
            pos, c32 = pos[keep], c32[keep]
            order = np.lexsort((pos, -c32.astype(np.float64)))
            want = np.sort(pos[order[:k]])
            assert count[b] == len(want) == min(k, len(pos))
            assert np.array_equal(idx[b, :count[b]], want)


def test_slowfast_slow_select_invariants():
    """Every selected candidate is at least as confident as every candidate
    left out, and a tie at the boundary goes to the lower position."""
    rng = np.random.default_rng(6)
    conf = rng.integers(0, 4, (4, 64)).astype(np.float64) / 4
    idx, count = oracle.slowfast_slow_select(conf, None, [0, 10, 30, 60], 32, 5)
    for b, st in enumerate([0, 10, 30, 60]):
        window = set(range(st, min(st + 32, 64)))
        sel = set(idx[b, :count[b]].tolist())
        rest = window - sel
        assert count[b] == min(5, len(window))
        if sel and rest:
            lo = min(conf[b, p] for p in sel)
            assert all(conf[b, p] <= lo for p in rest)
            assert all(p > max(q for q in sel if conf[b, q] == lo)
                       for p in rest if conf[b, p] == lo)


def test_slowfast_fast_select_against_boolean_masks():
    """The fast phase equals numpy's boolean selection of the masked region
    positions above the threshold, and its special cases: tau = -inf takes
    every masked non-NaN position of the region, a region ending at or
    before its start and a threshold of 1 (conf <= 1) take none."""
    rng = np.random.default_rng(7)
    B, L = 5, 400
    conf = rng.random((B, L))
    conf[rng.random((B, L)) < 0.03] = np.nan
    masked = (rng.random((B, L)) < 0.8).astype(np.uint8)
    start = rng.integers(0, L, B)
    end = np.minimum(start + rng.integers(0, 200, B), L)
    for tau in (0.3, 0.9, -np.inf, 1.0):
        idx, count = oracle.slowfast_fast_select(conf, masked, start, end, tau)
        for b in range(B):
            region = np.zeros(L, dtype=bool)
            region[start[b]:end[b]] = True
            want = np.flatnonzero(region & (masked[b] != 0) &
                                  (conf[b].astype(np.float32) > np.float32(tau)))
            assert np.array_equal(idx[b, :count[b]], want)
            if tau == 1.0:
                assert count[b] == 0
    idx, count = oracle.slowfast_fast_select(conf, masked, [50] * B, [50] * B, 0.0)
    assert count.tolist() == [0] * B
