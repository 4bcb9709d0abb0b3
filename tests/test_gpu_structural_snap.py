"""GPU parity of LSP's structural snapping of the committed block.

LSP, technical summary section 2, step 3: the block ends after its last
boundary token at or beyond the minimum length; lengths are integers, so they
are compared bit-exactly with the oracle on the same tokens.
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


@pytest.mark.parametrize("min_len", [0, 1, 17, 600])
def test_snap_matches_oracle(dl, min_len):
    g = torch.Generator().manual_seed(min_len + 1)
    B, L, V = 6, 3000, 126464
    tokens = torch.randint(0, V, (B, L), generator=g, dtype=torch.int32)
    delim = (torch.rand(V, generator=g) < 0.005).to(torch.uint8)
    # make boundaries frequent enough in the blocks: every 40th position on
    # average holds one of the boundary ids
    ids = torch.nonzero(delim)[:, 0].int()
    plant = torch.rand((B, L), generator=g) < 0.025
    tokens[plant] = ids[torch.randint(0, len(ids), (int(plant.sum()),), generator=g)]
    start = torch.tensor([0, 5, 1000, 2999, 3000, 1234], dtype=torch.int32)
    length = torch.tensor([3000, 700, 1500, 1, 0, 0], dtype=torch.int32)
    got = length.clone().cuda()
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    dl.dllm_snap_prefix(tokens.cuda(), delim.cuda(), start.cuda(), got, min_len=min_len,
                        dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    ref = oracle.snap_prefix(tokens.numpy(), delim.numpy(), start.numpy(), length.numpy(),
                             min_len)
    assert np.array_equal(got.cpu().numpy(), ref)
    if min_len <= 17:
        assert np.any(ref != length.numpy())  # some blocks do move


def test_adaptive_prefix_then_snap(dl):
    """The adaptive prefix on margin-like scores, then snapping on argmax
    tokens, both on the GPU; each compared with the oracle on the GPU's own
    inputs to that call."""
    g = torch.Generator().manual_seed(9)
    B, L, V = 4, 2048, 1000
    score = (torch.rand((B, L), generator=g) + torch.linspace(3, 0, L)[None, :]).float()
    tokens = torch.randint(0, V, (B, L), generator=g, dtype=torch.int32)
    delim = torch.zeros(V, dtype=torch.uint8)
    delim[[3, 14, 159]] = 1
    tokens[torch.rand((B, L), generator=g) < 0.05] = 14
    start = torch.tensor([0, 100, 1024, 2000], dtype=torch.int32)
    length, tau = dl.dllm_adaptive_prefix(score.cuda(), start.cuda(), 0.25, 0.5)
    snapped = length.clone()
    k_lo = 32
    dl.dllm_snap_prefix(tokens.cuda(), delim.cuda(), start.cuda(), snapped, min_len=k_lo)
    torch.cuda.synchronize()
    ref_len, _ = oracle.adaptive_prefix(score.numpy(), start.numpy(), 0.25, 0.5)
    assert np.array_equal(length.cpu().numpy(), ref_len)
    ref = oracle.snap_prefix(tokens.numpy(), delim.numpy(), start.numpy(), ref_len, k_lo)
    assert np.array_equal(snapped.cpu().numpy(), ref)


def test_snap_flags_bad_blocks_and_tokens(dl):
    tokens = torch.zeros((2, 10), dtype=torch.int32, device="cuda")
    tokens[1, 3] = 99  # outside the vocabulary of 8
    delim = torch.ones(8, dtype=torch.uint8, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    length = torch.tensor([11, 5], dtype=torch.int32, device="cuda")  # row 0 runs past L
    dl.dllm_snap_prefix(tokens, delim, torch.tensor([0, 0], dtype=torch.int32, device="cuda"),
                        length, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) != 0
    assert int(length[0]) == 11  # left as it was
    assert int(length[1]) == 5   # position 4 is a boundary: the block keeps its end
