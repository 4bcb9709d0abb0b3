"""The block-wise decoding loop, step after step, against the float64 oracle.

State carries from step to step on both sides: the K/V cache written by
earlier steps, the per-position score (the confidence of each position's
latest prediction) and ``start``, which every step's prefix commit advances.
Each step is checked before the next one runs: selection and compaction
bit-exact (decided on the GPU's own cosines, and equal to the planted set),
the whole cache bit-exact, attention and column sums (all heads on the small
loop, sampled heads at full size; column-sum row sums on every head), the
confidence, argmax and margin of every active row, the prefix length
bit-exact on the GPU's score and on the oracle's own, and ``start``.  The
first steps of the 128-step loop run in the launch configuration the bench
times, including two steps whose window is the whole sequence.
"""
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


class OracleLoop:
    """The oracle's side of the loop: cache, score and start carried in float64."""

    def __init__(self, shape, pools):
        self.s = shape
        self.kc = f64(pools["k_cache"])
        self.vc = f64(pools["v_cache"])
        self.prev = f64(pools["prev"])
        self.score = np.zeros((shape.B, shape.L))
        self.score[:, :shape.prompt] = np.inf
        self.start = np.full(shape.B, shape.prompt, dtype=np.int64)


def run_and_check(dl, shape, n_steps, heads_per_row):
    pools = workloads.make_loop_pools(shape)
    cap = workloads.loop_row_cap(shape)
    dev_pools = {k: v.cuda() for k, v in pools.items()}
    lp = dl.BlockDecodeLoop(shape.B, shape.L, shape.H, shape.d, shape.V, shape.dtype,
                            shape.prompt, cap, shape.tau, shape.tau_c)
    lp.reset(dev_pools["k_cache"], dev_pools["v_cache"])
    ref = OracleLoop(shape, pools)
    g = torch.Generator().manual_seed(99)
    for s in range(n_steps):
        inp = workloads.loop_step_inputs(shape, pools, s, cap)          # CPU, for the oracle
        dinp = workloads.loop_step_inputs(shape, dev_pools, s, cap)     # the same bits, built on the GPU
        for k in ("cur", "q", "k_new", "v_new", "logits"):
            assert torch.equal(inp[k], dinp[k].cpu()), (s, k)
        w = inp["win_start"]
        Lw = shape.L - w
        score_before = f64(lp.score)
        lp.step(dinp["cur"], dev_pools["prev"], dinp["q"], dinp["k_new"], dinp["v_new"],
                dinp["logits"], w)
        torch.cuda.synchronize()
        assert int(lp.dev_status[0]) == 0, s

        # selection: cosines; compaction of the GPU's cosines; the planted set
        cur = f64(inp["cur"])
        ref_cos = oracle.saliency_cos(cur[:, w:], ref.prev[:, w:])
        gcos = i32(lp.cos(Lw))
        assert np.max(np.abs(gcos - ref_cos)) <= SCORE_TOL, s
        idx, count = oracle.compact(oracle.salient_flags(gcos, shape.tau), w)
        assert np.array_equal(i32(lp.count), count), s
        assert np.array_equal(i32(lp.idx(Lw)), idx), s
        _, own_idx, own_count = oracle.saliency_select(cur[:, w:], ref.prev[:, w:], shape.tau,
                                                       idx_base=w)
        assert np.array_equal(own_idx, idx) and np.array_equal(own_count, count), s
        for b in range(shape.B):
            assert np.array_equal(idx[b, :count[b]], inp["planted"][b].numpy()), (s, b)
        # the cache, bit-exact, with every earlier step's rows in it
        ref.kc, ref.vc = oracle.kv_scatter(ref.kc, ref.vc, f64(inp["k_new"]), f64(inp["v_new"]),
                                           idx, count)
        assert np.array_equal(f64(lp.k_cache), ref.kc), s
        assert np.array_equal(f64(lp.v_cache), ref.vc), s
        # attention and column sums
        go, gl, gc = f64(lp.o), f64(lp.lse), f64(lp.colsum)
        q = f64(inp["q"])
        for b in range(shape.B):
            n = int(count[b])
            hs = range(shape.H) if heads_per_row is None else \
                torch.randperm(shape.H, generator=g)[:heads_per_row].tolist()
            for h in hs:
                ro, rl, rc = oracle.partial_attention(q[b:b + 1, :, h:h + 1],
                                                      ref.kc[b:b + 1, :, h:h + 1],
                                                      ref.vc[b:b + 1, :, h:h + 1], [n])
                r = ro[0, :n, 0]
                assert np.all(np.abs(go[b, :n, h] - r) <= BF16_ATOL + BF16_RTOL * np.abs(r)), \
                    (s, b, h)
                assert np.max(np.abs(gl[b, h, :n] - rl[0, 0, :n])) <= SCORE_TOL, (s, b, h)
                assert np.max(np.abs(gc[b, h] - rc[0, 0])) <= SCORE_TOL, (s, b, h)
            assert np.max(np.abs(gc[b].sum(-1) - n)) <= 1e-4 * max(n, 1), (s, b)
        # confidence of every active row, at its position
        rcf, ram, rmg = oracle.confidence(f64(inp["logits"]), count=count)
        gsc, gam, gmg = f64(lp.score), i32(lp.argmax), f64(lp.margin)
        written = np.zeros((shape.B, shape.L), dtype=bool)
        for b in range(shape.B):
            n = int(count[b])
            pos = idx[b, :n]
            assert np.all(np.abs(gsc[b, pos] - rcf[b, :n]) <= 1e-6 + SCORE_TOL * np.abs(rcf[b, :n])), \
                (s, b)
            assert np.array_equal(gam[b, pos], ram[b, :n]), (s, b)
            assert np.max(np.abs(gmg[b, pos] - rmg[b, :n])) <= 1e-6, (s, b)
            ref.score[b, pos] = rcf[b, :n]
            written[b, pos] = True
        assert np.array_equal(gsc[~written], score_before[~written]), s  # the rest untouched
        # prefix commit: on the GPU's score and on the oracle's own, from the same start
        glen = i32(lp.length)
        assert np.array_equal(glen, oracle.stable_prefix(gsc.astype(np.float32), ref.start,
                                                         shape.tau_c, True)), s
        assert np.array_equal(glen, oracle.stable_prefix(ref.score, ref.start, shape.tau_c, True)), s
        ref.start = ref.start + glen
        assert np.array_equal(i32(lp.start), ref.start), s
        # the schedule's commit: the block's next positions, every step
        assert glen.tolist() == [shape.commit] * shape.B, (s, glen)


def test_small_loop_all_steps(dl):
    """Four blocks of 32 (16 steps, four of them over the whole sequence), every head."""
    run_and_check(dl, workloads.LOOP_SMALL, workloads.LOOP_SMALL.T, None)


def test_loop_128_first_steps_full_size(dl):
    """The first 8 steps of the batch-4 L 2048 loop (steps 0 and 4 over all 2048 rows)."""
    run_and_check(dl, workloads.LOOP_128, 8, 2)
