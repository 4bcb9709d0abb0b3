"""GPU parity of the approximate output update of the stable rows.

DyLLM, technical summary, Methodology 2 (non-salient path): the outputs of
stable rows move by the value changes of the salient rows weighted by the
previous step's attention weights.  Compared with the float64 oracle on the
same inputs: within 1e-4 for float32 (float32 dot products of up to 128 terms
and sums over up to 410 salient columns), within 2e-2 + 1e-2 |ref| for
bfloat16 outputs (one rounding of the updated output to bfloat16); rows that
are not listed as stable stay bitwise unchanged.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

F32_ATOL = 1e-4
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


def _sets(g, B, L, counts, M_max, N_max):
    """Salient positions (ascending) and the stable rest, per batch row."""
    idx = torch.full((B, M_max), -1, dtype=torch.int32)
    stable = torch.full((B, N_max), -1, dtype=torch.int32)
    s_counts = []
    for b in range(B):
        perm = torch.randperm(L, generator=g)
        idx[b, :counts[b]] = torch.sort(perm[:counts[b]]).values.int()
        rest = torch.sort(perm[counts[b]:]).values[:N_max].int()
        stable[b, :len(rest)] = rest
        s_counts.append(len(rest))
    return idx, torch.tensor(counts, dtype=torch.int32), stable, torch.tensor(s_counts,
                                                                             dtype=torch.int32)


def _run(dl, q, lse, k, v, v_new, idx, count, stable, s_count, o, scale=0.0, st=None):
    c = lambda t: t.cuda()  # noqa: E731
    out = c(o)
    dl.dllm_approx_attention_update(c(q), c(lse), c(k), c(v), c(v_new), c(idx), c(count),
                                    c(stable), c(s_count), out, scale=scale, dev_status=st)
    torch.cuda.synchronize()
    return out


def _untouched(out, o, stable, s_count):
    B, L = o.shape[:2]
    mask = np.ones((B, L), dtype=bool)
    for b in range(B):
        mask[b, stable[b, :int(s_count[b])].numpy()] = False
    return np.array_equal(f64(out)[mask], f64(o)[mask])


@pytest.mark.parametrize("d", [32, 64, 128])
def test_update_float32_exact_identity(dl, d):
    """Queries and keys unchanged, values changed at the salient positions:
    the update equals attention recomputed over the new values."""
    g = torch.Generator().manual_seed(d)
    B, L, H = 2, 300, 2
    q, k, v = (torch.randn((B, L, H, d), generator=g) for _ in range(3))
    o_ref, lse_ref, _ = oracle.partial_attention(f64(q), f64(k), f64(v), [L] * B)
    o = torch.from_numpy(o_ref).float()
    lse = torch.from_numpy(lse_ref).float()
    idx, count, stable, s_count = _sets(g, B, L, [70, 130], 160, 300)
    v_new = torch.randn((B, 160, H, d), generator=g)
    out = _run(dl, q, lse, k, v, v_new, idx, count, stable, s_count, o)
    ref = oracle.approx_attention_update(f64(o), f64(q), f64(lse), f64(k), f64(v), f64(v_new),
                                         idx.numpy(), count.numpy(), stable.numpy(),
                                         s_count.numpy())
    assert np.max(np.abs(f64(out) - ref)) <= F32_ATOL
    assert _untouched(out, o, stable, s_count)
    # and the identity itself, on the GPU's result
    _, v_upd = oracle.kv_scatter(f64(k), f64(v), f64(k), f64(v_new), idx.numpy(), count.numpy())
    o_exact, _, _ = oracle.partial_attention(f64(q), f64(k), v_upd, [L] * B)
    for b in range(B):
        rows = stable[b, :int(s_count[b])].numpy()
        assert np.max(np.abs(f64(out)[b, rows] - o_exact[b, rows])) <= 2 * F32_ATOL


def test_update_bf16_full_size(dl):
    """B1, L4096, 32 heads of 128, 410 salient positions, every other
    position stable."""
    g = torch.Generator().manual_seed(7)
    B, L, H, d, n_sal = 1, 4096, 32, 128, 410
    bf = torch.bfloat16
    q, k, v = (torch.randn((B, L, H, d), generator=g).to(bf) for _ in range(3))
    o = (0.5 * torch.randn((B, L, H, d), generator=g)).to(bf)
    # log-sum-exps below log L make the weights, and so the update, large
    # against the bfloat16 rounding of the outputs
    lse = (math.log(L) - 4.0 + 0.25 * torch.randn((B, H, L), generator=g)).float()
    idx, count, stable, s_count = _sets(g, B, L, [n_sal], n_sal, L)
    v_new = torch.randn((B, n_sal, H, d), generator=g).to(bf)
    out = _run(dl, q, lse, k, v, v_new, idx, count, stable, s_count, o)
    ref = oracle.approx_attention_update(f64(o), f64(q), f64(lse), f64(k), f64(v), f64(v_new),
                                         idx.numpy(), count.numpy(), stable.numpy(),
                                         s_count.numpy())
    got = f64(out)
    assert np.all(np.abs(got - ref) <= BF16_ATOL + BF16_RTOL * np.abs(ref)), np.max(np.abs(got - ref))
    # the update itself agrees to within the rounding of the outputs
    du_ref, du_got = ref - f64(o), got - f64(o)
    assert np.linalg.norm(du_got - du_ref) <= 0.03 * np.linalg.norm(du_ref)
    assert np.std(du_ref) > 0.2
    assert _untouched(out, o, stable, s_count)


def test_update_edge_cases(dl):
    g = torch.Generator().manual_seed(3)
    B, L, H, d = 2, 100, 2, 64
    q, k, v = (torch.randn((B, L, H, d), generator=g) for _ in range(3))
    o = torch.randn((B, L, H, d), generator=g)
    lse = torch.full((B, H, L), 5.0)
    idx, count, stable, s_count = _sets(g, B, L, [10, 0], 16, 64)
    v_new = torch.randn((B, 16, H, d), generator=g)
    # batch row 1 has no salient position: its outputs stay as they are
    out = _run(dl, q, lse, k, v, v_new, idx, count, stable, s_count, o, scale=0.2)
    ref = oracle.approx_attention_update(f64(o), f64(q), f64(lse), f64(k), f64(v), f64(v_new),
                                         idx.numpy(), count.numpy(), stable.numpy(),
                                         s_count.numpy(), scale=0.2)
    assert np.max(np.abs(f64(out) - ref)) <= F32_ATOL
    assert np.array_equal(f64(out)[1], f64(o)[1])
    # no stable row: nothing changes
    out = _run(dl, q, lse, k, v, v_new, idx, count, stable, torch.zeros(B, dtype=torch.int32), o)
    assert torch.equal(out.cpu(), o)
    # a stable position out of range is flagged and skipped
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    bad = stable.clone()
    bad[0, 0] = L + 5
    out = _run(dl, q, lse, k, v, v_new, idx, count, bad, s_count, o, st=st)
    assert int(st[0]) != 0


@pytest.mark.parametrize("counts", [[1, 129], [128, 0], [257, 64]])
def test_update_bf16_tensor_cores_ragged(dl, counts):
    """bf16 with head dim 128 (the tensor-core kernel): salient counts on
    both sides of the 128-column passes, a batch row with none, stable lists
    that leave rows out and end in a ragged tile; against the oracle, rows
    outside the lists bitwise unchanged, and the exact identity when only
    values change."""
    g = torch.Generator().manual_seed(sum(counts))
    B, L, H, d = 2, 700, 4, 128
    bf = torch.bfloat16
    q, k, v = (torch.randn((B, L, H, d), generator=g).to(bf) for _ in range(3))
    o_ref, lse_ref, _ = oracle.partial_attention(f64(q), f64(k), f64(v), [L] * B)
    o = torch.from_numpy(o_ref).to(bf)
    lse = torch.from_numpy(lse_ref).float()
    idx, count, stable, s_count = _sets(g, B, L, counts, 300, 450)
    v_new = torch.randn((B, 300, H, d), generator=g).to(bf)
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    out = _run(dl, q, lse, k, v, v_new, idx, count, stable, s_count, o, st=st)
    assert int(st[0]) == 0
    ref = oracle.approx_attention_update(f64(o), f64(q), f64(lse), f64(k), f64(v), f64(v_new),
                                         idx.numpy(), count.numpy(), stable.numpy(),
                                         s_count.numpy())
    got = f64(out)
    assert np.all(np.abs(got - ref) <= BF16_ATOL + BF16_RTOL * np.abs(ref)), np.max(np.abs(got - ref))
    assert _untouched(out, o, stable, s_count)
    if counts[1] == 0:
        assert torch.equal(out[1].cpu(), o[1])
    # the identity: attention recomputed over the updated values (float64 on
    # the same bf16 inputs), to within the bf16 rounding of the outputs
    _, v_upd = oracle.kv_scatter(f64(k), f64(v), f64(k), f64(v_new), idx.numpy(), count.numpy())
    o_exact, _, _ = oracle.partial_attention(f64(q), f64(k), v_upd, [L] * B)
    for b in range(B):
        rows = stable[b, :int(s_count[b])].numpy()
        e = o_exact[b, rows]
        assert np.all(np.abs(got[b, rows] - e) <= BF16_ATOL + BF16_RTOL * np.abs(e))
