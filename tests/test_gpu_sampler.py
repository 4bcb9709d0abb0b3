"""GPU parity of the attention-guided decoding order (Attn-Sampler).

Attn-Sampler, technical summary, Methodology 1 and 2: total attention per
position (the column sums summed over heads, and over layers by
accumulation) within 1e-5 relative of the float64 oracle (float32 adds of
32 non-negative terms); the order and the count of tokens to decode
bit-exactly against the oracle's decision taken on the GPU's own float32
scores (the decision is a float32 compare on both sides).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

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


def test_scores_sum_heads_and_accumulate(dl):
    g = torch.Generator().manual_seed(11)
    B, H, L = 3, 32, 1000
    colsum = torch.rand((B, H, L), generator=g) * 3.0
    a = dl.dllm_attn_scores(colsum.cuda())
    torch.cuda.synchronize()
    ref = oracle.attn_scores(colsum.double().numpy())
    got = a.cpu().double().numpy()
    assert np.max(np.abs(got - ref) / np.maximum(ref, 1e-30)) <= 1e-5
    a2 = dl.dllm_attn_scores(colsum.cuda(), score_inout=a.clone(), accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(a2.cpu(), 2 * a.cpu())  # s + s is exact


def _check_select(dl, score, cand, tau, gamma, k_max):
    order, n = dl.dllm_attn_sampler_select(score.cuda(),
                                           candidates=None if cand is None else cand.cuda(),
                                           tau=tau, gamma=gamma, k_max=k_max)
    torch.cuda.synchronize()
    ro, rn = oracle.attn_sampler_select(score.numpy(), None if cand is None else cand.numpy(),
                                        tau, gamma, k_max)
    assert np.array_equal(order.cpu().numpy(), ro)
    assert np.array_equal(n.cpu().numpy(), rn)
    return rn


@pytest.mark.parametrize("L", [1, 7, 1000, 1024, 4096, 16384])
def test_select_matches_oracle(dl, L):
    g = torch.Generator().manual_seed(L)
    B = 3
    score = torch.round(torch.rand((B, L), generator=g) * 64) / 64  # many ties
    cand = (torch.rand((B, L), generator=g) < 0.6).to(torch.uint8)
    cand[2] = 0  # a batch row with no candidate
    for tau, gamma, k_max in [(0.0, 0.0, 0), (0.5, 0.0, 0), (0.0, 0.9, 0), (0.2, 0.5, 8),
                              (2.0, 0.0, 0), (0.0, 1.0, 0)]:
        rn = _check_select(dl, score, cand, tau, gamma, k_max)
        assert rn[2] == 0


def test_select_special_values(dl):
    score = torch.tensor([[float("nan"), 0.0, -0.0, 1.0, float("-inf"), float("inf"), 1.0]])
    for tau, gamma in [(-1.0, 0.0), (0.0, 0.5), (0.5, 1.0)]:
        _check_select(dl, score, None, tau, gamma, 0)


def test_colsum_to_order_chain(dl):
    """Column sums of the partial attention, summed over heads on the GPU,
    ordered on the GPU: the order is the oracle's on the GPU's scores, the
    scores are the oracle's column sums summed over heads."""
    s = workloads.TINY_F32
    inp = workloads.make_step(s, n_salient=s.L, with_logits=False)
    count = torch.full((s.B,), s.L, dtype=torch.int32)
    o, lse, cs = dl.dllm_partial_attention(inp["q"].cuda(), inp["k_cache"].cuda(),
                                           inp["v_cache"].cuda(), count.cuda())
    a = dl.dllm_attn_scores(cs)
    order, n = dl.dllm_attn_sampler_select(a, tau=0.0, gamma=0.5)
    torch.cuda.synchronize()
    _, _, rcs = oracle.partial_attention(inp["q"].double().numpy(), inp["k_cache"].double().numpy(),
                                         inp["v_cache"].double().numpy(), count.numpy())
    ref_a = oracle.attn_scores(rcs)
    assert np.max(np.abs(a.cpu().double().numpy() - ref_a)) <= 1e-4
    ro, rn = oracle.attn_sampler_select(a.cpu().numpy(), None, 0.0, 0.5, 0)
    assert np.array_equal(order.cpu().numpy(), ro) and np.array_equal(n.cpu().numpy(), rn)


def test_sampler_errors(dl):
    s = torch.zeros((1, 16), device="cuda")
    with pytest.raises(RuntimeError):
        dl.dllm_attn_sampler_select(s, tau=float("nan"))
    with pytest.raises(RuntimeError):
        dl.dllm_attn_sampler_select(torch.zeros((1, 16385), device="cuda"))
