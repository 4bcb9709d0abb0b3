"""Host side of the block-wise decoding loop (CPU): its schedule and inputs.

The schedule is checked against what the loop is meant to do, with the
float64 oracle playing every step of the small loop: each step selects
exactly its planted set, and the prefix commit takes exactly the block's next
``commit`` positions, so ``start`` walks through the generated positions one
block per ``steps_per_block`` steps.
"""
import numpy as np
import torch

import oracle
import workloads


def test_schedule_constants():
    s = workloads.LOOP_128
    assert s.T == 128
    assert (s.L - s.prompt) // s.block == 32
    assert s.block == s.commit * s.steps_per_block
    assert [workloads.loop_window(s, t) for t in range(8)] == [0, 1024, 1024, 1024] * 2
    assert workloads.loop_block(s, 0) == (1024, 0)
    assert workloads.loop_block(s, 127) == (2048 - 32, 3)
    assert workloads.loop_undecoded(s, 5) == (1024 + 32 + 8, 1024 + 64)
    assert workloads.loop_boosted(s, 6) == (1024 + 32, 1024 + 32 + 24)


def test_planted_sets():
    s = workloads.LOOP_128
    counts = workloads.loop_counts(s)
    assert counts.shape == (s.T, s.B)
    for t in (0, 1, 2, 3, 64, 127):
        lo, hi = workloads.loop_undecoded(s, t)
        for p in workloads.loop_planted(s, t):
            p = p.numpy()
            assert np.all(np.diff(p) > 0)                      # sorted, distinct
            assert np.all((p >= s.prompt) & (p < s.L))         # generated positions only
            assert set(range(lo, hi)) <= set(p.tolist())       # the block's undecoded rows
            assert s.n_random <= len(p) <= s.n_random + (hi - lo)
    # a per-step generator: the same step gives the same set, in any order of calls
    a = [x.clone() for x in workloads.loop_planted(s, 17)]
    workloads.loop_planted(s, 3)
    assert all(torch.equal(x, y) for x, y in zip(a, workloads.loop_planted(s, 17)))
    assert workloads.loop_row_cap(s) == int(counts.max())


def test_step_inputs_layout():
    s = workloads.LOOP_SMALL
    pools = workloads.make_loop_pools(s)
    cap = workloads.loop_row_cap(s)
    for t in (0, 1, 7):
        inp = workloads.loop_step_inputs(s, pools, t, cap)
        w = inp["win_start"]
        assert inp["q"].shape == (s.B, cap, s.H, s.d)
        assert inp["k_new"].shape == (s.B, s.L - w, s.H, s.d)
        assert inp["logits"].shape == (s.B, cap, s.V)
        blo, bhi = workloads.loop_boosted(s, t)
        for b in range(s.B):
            pl = inp["planted"][b]
            n = len(pl)
            hot = torch.zeros(s.L, dtype=torch.bool)
            hot[pl] = True
            assert torch.equal(inp["cur"][b][hot], pools["hot"][b][hot])
            assert torch.equal(inp["cur"][b][~hot], pools["cold"][b][~hot])
            assert torch.count_nonzero(inp["q"][b, n:]) == 0
            assert torch.count_nonzero(inp["logits"][b, n:]) == 0
            # boosted rows: one logit raised by the boost (in float64, then cast)
            raised = (inp["logits"][b, :n].double() - 0).max(-1).values
            for r in range(n):
                is_boost = blo <= int(pl[r]) < bhi
                assert (raised[r] > 10.0) == is_boost, (t, b, r)


def test_oracle_plays_the_small_loop():
    """Every step of the small loop under the oracle: the planted set is
    selected and exactly ``commit`` positions are committed."""
    s = workloads.LOOP_SMALL
    pools = workloads.make_loop_pools(s)
    cap = workloads.loop_row_cap(s)
    f = lambda t: t.double().numpy()  # noqa: E731
    kc, vc, prev = f(pools["k_cache"]), f(pools["v_cache"]), f(pools["prev"])
    score = np.zeros((s.B, s.L))
    score[:, :s.prompt] = np.inf
    start = np.full(s.B, s.prompt)
    for t in range(s.T):
        inp = workloads.loop_step_inputs(s, pools, t, cap)
        w = inp["win_start"]
        _, idx, count = oracle.saliency_select(f(inp["cur"])[:, w:], prev[:, w:], s.tau,
                                               idx_base=w)
        for b in range(s.B):
            assert np.array_equal(idx[b, :count[b]], inp["planted"][b].numpy())
        kc, vc = oracle.kv_scatter(kc, vc, f(inp["k_new"]), f(inp["v_new"]), idx, count)
        o, lse, colsum = oracle.partial_attention(f(inp["q"]), kc, vc, count)
        assert np.allclose(colsum.sum(-1), count[:, None])
        conf, _, _ = oracle.confidence(f(inp["logits"]), count=count)
        for b in range(s.B):
            score[b, idx[b, :count[b]]] = conf[b, :count[b]]
        ln = oracle.stable_prefix(score, start, s.tau_c, True)
        assert ln.tolist() == [s.commit] * s.B, (t, ln)
        assert start.tolist() == [workloads.loop_undecoded(s, t)[0]] * s.B
        start = start + ln
    assert start.tolist() == [s.L] * s.B
