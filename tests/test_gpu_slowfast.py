"""SlowFast sampling on the GPU against the float64 oracle.

The device controller (dllm_slowfast_observe_device) must report exactly the
phases and region ends of oracle.slowfast_phases over long random prediction
sequences; the token selection (dllm_slowfast_select) exactly the positions
and counts of oracle.slowfast_select on the same float32 confidences (ties,
NaN, masks, windows cut at L, regions at the ends); and a device-resident
chain of steps -- stable prefix of the confidences as the convergence
prediction, the controller, the selection, the unmasking -- must follow the
oracle step by step.

SlowFast, section 2 (pipeline: exploratory phase, variance of e_cand below
sigma^2_stable, accelerated phase over [s_cycle, e_cycle]).
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from partial_attention_saliency_b300 import build
    build.build_library()
    import partial_attention_saliency_b300 as dl
    dl.load_library()
    return dl


@pytest.mark.parametrize("window,sigma2", [(1, 0.5), (3, 0.25), (3, 2.0 / 9.0), (5, 3.5),
                                           (8, 40.0), (2, 0.0)])
def test_device_controller_matches_oracle(dl, window, sigma2):
    rng = np.random.default_rng(window * 131 + int(sigma2 * 7))
    B, T = 6, 300
    steps = rng.choice([0, 0, 0, 1, 2, 7], size=(T, B))
    e = (np.cumsum(steps, axis=0) + rng.integers(0, 2, (T, B))).astype(np.int32)
    starts = np.maximum(e - rng.integers(0, 6, (T, B)), 0).astype(np.int32)
    ref_phase, ref_end = oracle.slowfast_phases(starts, e, window, sigma2)
    sf = dl.SlowFastDevice(B, window, sigma2)
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    for t in range(T):
        s_dev = torch.from_numpy(starts[t]).cuda()
        l_dev = torch.from_numpy(e[t] - starts[t]).cuda()
        phase, end = sf.observe(s_dev, l_dev, dev_status=st)
        assert np.array_equal(phase.cpu().numpy(), ref_phase[t]), t
        assert np.array_equal(end.cpu().numpy(), ref_end[t]), t
    assert int(st[0]) == 0
    if sigma2 > 1.0 and window <= 5:
        assert ref_phase.sum() > 0


@pytest.mark.parametrize("L,width,k", [(1, 1, 1), (300, 64, 1), (300, 300, 5), (5000, 1024, 64),
                                       (20000, 16384, 37), (1000, 16384, 64)])
def test_select_matches_oracle(dl, L, width, k):
    rng = np.random.default_rng(L + width + k)
    B = 8
    conf = np.round(rng.random((B, L)), 2).astype(np.float32)   # many ties
    conf[rng.random((B, L)) < 0.03] = np.nan
    conf[0, :min(L, 5)] = -0.0
    masked = (rng.random((B, L)) < 0.75).astype(np.uint8)
    start = rng.integers(0, L + 1, B).astype(np.int32)
    start[1] = 0
    start[2] = L                                                  # nothing left
    phase = (rng.random(B) < 0.5).astype(np.int32)
    phase[3], phase[4] = 1, 0
    end = np.minimum(start + rng.integers(0, 2 * width + 1, B), L).astype(np.int32)
    end[5] = start[5]                                             # empty fast region
    for tau in (0.5, 0.9, -np.inf):
        for use_mask in (True, False):
            m = masked if use_mask else None
            ref_idx, ref_cnt = oracle.slowfast_select(conf.astype(np.float64), m, start, phase,
                                                      end, tau, width, k)
            st = torch.zeros((1,), dtype=torch.int32, device="cuda")
            idx, cnt = dl.dllm_slowfast_select(
                torch.from_numpy(conf).cuda(), torch.from_numpy(start).cuda(),
                torch.from_numpy(phase).cuda(), torch.from_numpy(end).cuda(), tau, width, k,
                masked=None if m is None else torch.from_numpy(m).cuda(), dev_status=st)
            torch.cuda.synchronize()
            assert int(st[0]) == 0
            assert np.array_equal(cnt.cpu().numpy(), ref_cnt), (tau, use_mask)
            assert np.array_equal(idx.cpu().numpy(), ref_idx), (tau, use_mask)


def test_select_flags_bad_start_and_region(dl):
    conf = torch.rand((2, 50), device="cuda")
    start = torch.tensor([60, 10], dtype=torch.int32, device="cuda")   # row 0: start > L
    phase = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    end = torch.tensor([0, 80], dtype=torch.int32, device="cuda")      # row 1: end > L, clamped
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    idx, cnt = dl.dllm_slowfast_select(conf, start, phase, end, -1.0, 8, 2, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 4  # DLLM_ERR_DEVICE_CHECK
    assert cnt.cpu().tolist() == [0, 40]
    assert idx[1, :40].cpu().tolist() == list(range(10, 50))


def test_device_resident_slowfast_steps(dl):
    """Steps of a SlowFast decode kept on the device: each step's convergence
    prediction is the stable prefix of the confidences (threshold tau_c) from
    start, the device controller decides the phase, the selection unmasks
    tokens (their confidence becomes +inf, so the prefix moves past them);
    the host only checks the results against the oracle."""
    rng = np.random.default_rng(17)
    B, L, W, sigma2 = 4, 512, 3, 2.0
    tau_c, tau_high, width, k = 0.7, 0.8, 32, 2
    conf_h = np.zeros((B, L), dtype=np.float32)
    masked_h = np.ones((B, L), dtype=np.uint8)
    start_h = np.zeros(B, dtype=np.int32)
    sf = dl.SlowFastDevice(B, W, sigma2)
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    starts, preds = [], []
    for t in range(60):
        # fresh confidences of the masked positions: confident up to the
        # next multiple of 40 past the start, noise beyond it, so the
        # prediction settles and the fast phase takes the band
        band = ((start_h // 40) + 1) * 40
        for b in range(B):
            pos = np.arange(L)
            c = np.where(pos < band[b], 0.85 + 0.1 * rng.random(L), 0.6 * rng.random(L))
            conf_h[b] = np.where(masked_h[b] != 0, c, np.inf).astype(np.float32)
        conf = torch.from_numpy(conf_h).cuda()
        start = torch.from_numpy(start_h).cuda()
        ln = dl.dllm_stable_prefix(conf, start, tau_c, min_commit=False, advance_start=False,
                                   dev_status=st)
        phase, end = sf.observe(start, ln, dev_status=st)
        idx, cnt = dl.dllm_slowfast_select(conf, start, phase, end, tau_high, width, k,
                                           masked=torch.from_numpy(masked_h).cuda(), dev_status=st)
        torch.cuda.synchronize()
        assert int(st[0]) == 0
        # the oracle on the same step
        ref_len = oracle.stable_prefix(conf_h, start_h, tau_c, False)
        assert np.array_equal(ln.cpu().numpy(), ref_len), t
        starts.append(start_h.copy())
        preds.append(start_h + ref_len)
        ref_phase, ref_end = oracle.slowfast_phases(starts, preds, W, sigma2)
        assert np.array_equal(phase.cpu().numpy(), ref_phase[-1]), t
        assert np.array_equal(end.cpu().numpy(), ref_end[-1]), t
        ref_idx, ref_cnt = oracle.slowfast_select(conf_h, masked_h, start_h, ref_phase[-1],
                                                  ref_end[-1], tau_high, width, k)
        assert np.array_equal(cnt.cpu().numpy(), ref_cnt), t
        assert np.array_equal(idx.cpu().numpy(), ref_idx), t
        # unmask the selected tokens; start moves past the unmasked prefix
        for b in range(B):
            masked_h[b, ref_idx[b, :ref_cnt[b]]] = 0
            while start_h[b] < L and masked_h[b, start_h[b]] == 0:
                start_h[b] += 1
    assert ref_phase.sum() > 0 and (ref_phase == 0).sum() > 0  # both phases were taken
