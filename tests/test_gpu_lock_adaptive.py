"""GPU parity of the lock criterion and the adaptive prefix threshold.

SureLock, technical summary section 2, locking criteria 1 and 2: the local
KL divergence of each position's distribution between two steps and its
uncertainty, compared with the float64 oracle within 1e-4 (the float32
accumulation of up to 126464 exponentials, two log-sum-exps and one
difference of them); the lock flags are compared bit-exactly with the
oracle's decision taken on the GPU's own divergences and uncertainties (the
decision is a float32 compare on both sides).  LSP, technical summary
section 2, step 2: lengths and thresholds of the adaptive prefix are
bit-exact against the oracle on the same float32 scores.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

KL_ATOL, KL_RTOL = 1e-4, 1e-5
UNC_ATOL = 1e-5


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


def _pair(g, B, R, V, dtype, spread):
    """Current logits and previous ones that differ from them by noise of a
    per-row scale from 1e-3 to ``spread`` (so the divergences span decades)."""
    z = workloads.normal(g, (B, R, V), 2.0, torch.float32)
    scale = torch.logspace(-3, np.log10(spread), R)[None, :, None]
    y = z + scale * torch.randn((B, R, V), generator=g)
    return z.to(dtype), y.to(dtype)


def _check_kl(kl, unc, ref_kl, ref_unc, mask):
    g, r = f64(kl)[mask], ref_kl[mask]
    assert np.all(np.abs(g - r) <= KL_ATOL + KL_RTOL * np.abs(r)), np.max(np.abs(g - r))
    assert np.max(np.abs(f64(unc)[mask] - ref_unc[mask])) <= UNC_ATOL


@pytest.mark.parametrize("dtype,V", [(torch.float32, 301), (torch.float32, 4096),
                                     (torch.bfloat16, 1000), (torch.bfloat16, 126464)])
def test_lock_kl_dense(dl, dtype, V):
    g = torch.Generator().manual_seed(V)
    B, R = 2, 24
    z, y = _pair(g, B, R, V, dtype, 1.0)
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    kl, unc, _ = dl.dllm_lock_criterion(z.cuda(), y.cuda(), 0.0, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    ref_kl, ref_unc = oracle.lock_kl(f64(z), f64(y))
    _check_kl(kl, unc, ref_kl, ref_unc, np.ones((B, R), dtype=bool))
    assert float(ref_kl.min()) < 1e-3 and float(ref_kl.max()) > 0.3  # the spread is real


@pytest.mark.parametrize("B", [3, 65])
def test_lock_kl_ragged_counts(dl, B):
    # B <= 64: the persistent partial kernel over the valid rows; 65: one CTA
    # per row slot.  Counts from 0 to R, so many row slots are empty.
    g = torch.Generator().manual_seed(B)
    R, V = 9, 1000
    z, y = _pair(g, B, R, V, torch.bfloat16, 1.0)
    count = torch.tensor([(7 * b) % (R + 1) for b in range(B)], dtype=torch.int32)
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    kl, unc, _ = dl.dllm_lock_criterion(z.cuda(), y.cuda(), 0.0, count=count.cuda(), dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    ref_kl, ref_unc = oracle.lock_kl(f64(z), f64(y))
    mask = np.arange(R)[None, :] < count.numpy()[:, None]
    _check_kl(kl, unc, ref_kl, ref_unc, mask)


def test_lock_kl_identical_rows_give_zero(dl):
    g = torch.Generator().manual_seed(5)
    z = workloads.normal(g, (1, 8, 126464), 3.0, torch.bfloat16)
    kl, unc, _ = dl.dllm_lock_criterion(z.cuda(), z.clone().cuda(), 0.0)
    torch.cuda.synchronize()
    assert np.max(np.abs(f64(kl))) <= KL_ATOL
    _, ref_unc = oracle.lock_kl(f64(z), f64(z))
    assert np.max(np.abs(f64(unc) - ref_unc)) <= UNC_ATOL


@pytest.mark.parametrize("gate_q", [0.0, 0.3, 0.5, 1.0])
def test_lock_gather_scatter_and_flags(dl, gate_q):
    """Rows gathered by row index, results scattered to positions, ragged
    counts (one batch row empty), flags set where both criteria hold and
    never cleared."""
    g = torch.Generator().manual_seed(17)
    B, R_src, V, L, R_max = 3, 40, 126464, 300, 32
    z, y = _pair(g, B, R_src, V, torch.bfloat16, 2.0)
    count = torch.tensor([32, 0, 19], dtype=torch.int32)
    row_idx = torch.stack([torch.randperm(R_src, generator=g)[:R_max] for _ in range(B)]).int()
    out_idx = torch.stack([torch.randperm(L, generator=g)[:R_max] for _ in range(B)]).int()
    locked0 = (torch.rand((B, L), generator=g) < 0.1).to(torch.uint8)
    kl0 = torch.full((B, L), -7.0)
    locked = locked0.clone().cuda()
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ref_kl_rows, ref_unc_rows = oracle.lock_kl(f64(z), f64(y), count=count.numpy(),
                                               row_idx=row_idx.numpy())
    active = ~np.isnan(ref_kl_rows)
    eps = float(np.median(ref_kl_rows[active]))
    kl, unc, _ = dl.dllm_lock_criterion(z.cuda(), y.cuda(), eps, gate_q=gate_q, R_max=R_max,
                                        row_idx=row_idx.cuda(), count=count.cuda(),
                                        out_idx=out_idx.cuda(), out_cols=L,
                                        kl_out=kl0.clone().cuda(), unc_out=kl0.clone().cuda(),
                                        locked_inout=locked, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    gkl, gunc, glk = f64(kl), f64(unc), locked.cpu().numpy()
    # read the scattered results back in row order
    rkl = np.full((B, R_max), np.nan)
    runc = np.full((B, R_max), np.nan)
    for b in range(B):
        n = int(count[b])
        cols = out_idx[b, :n].numpy()
        rkl[b, :n], runc[b, :n] = gkl[b, cols], gunc[b, cols]
    _check_kl(torch.from_numpy(rkl), torch.from_numpy(runc), ref_kl_rows, ref_unc_rows, active)
    # positions that no active row writes are untouched
    written = np.zeros((B, L), dtype=bool)
    for b in range(B):
        written[b, out_idx[b, :int(count[b])].numpy()] = True
    assert np.all(gkl[~written] == -7.0) and np.all(gunc[~written] == -7.0)
    # flags: the oracle's decision on the GPU's own divergences, bit-exact
    dec = oracle.lock_decision(rkl.astype(np.float32), runc.astype(np.float32), count.numpy(),
                               eps, gate_q)
    exp = locked0.numpy().astype(bool).copy()
    for b in range(B):
        n = int(count[b])
        exp[b, out_idx[b, :n].numpy()] |= dec[b, :n]
    assert np.array_equal(glk.astype(bool), exp)
    assert dec.sum() > 0 and (~dec[active]).sum() > 0
    assert np.all(glk[locked0.numpy() == 1] == 1)


def test_lock_gate_percentile_ties(dl):
    """Identical rows tie in uncertainty: the k-th smallest is that value and
    the gate passes all of them; distinct rows then split at the percentile."""
    g = torch.Generator().manual_seed(23)
    V, R = 5000, 40
    base = workloads.normal(g, (1, 1, V), 2.0, torch.float32)
    z = base.repeat(1, R, 1)
    z[0, 20:] += torch.linspace(0, 3, 20)[:, None] * (torch.arange(V) == 7).float()[None, :]
    y = z.clone()
    locked = torch.zeros((1, R), dtype=torch.uint8, device="cuda")
    kl, unc, _ = dl.dllm_lock_criterion(z.cuda(), y.cuda(), 1e-3, gate_q=0.5, locked_inout=locked)
    torch.cuda.synchronize()
    dec = oracle.lock_decision(f64(kl).astype(np.float32), f64(unc).astype(np.float32), [R],
                               1e-3, 0.5)
    assert np.array_equal(locked.cpu().numpy().astype(bool), dec)
    assert dec[0, :20].all()


def test_lock_errors(dl):
    z = torch.zeros((1, 4, 64), device="cuda")
    with pytest.raises(RuntimeError):
        dl.dllm_lock_criterion(z, z, 0.1, ws=torch.empty((16,), dtype=torch.uint8, device="cuda"))
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    bad = torch.tensor([[0, 1, 9, 2]], dtype=torch.int32, device="cuda")  # row 9 out of range
    dl.dllm_lock_criterion(z, z, 0.1, row_idx=bad, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) != 0


# ------------------------------------------------------------ adaptive prefix

def _scores(g, B, L):
    s = torch.rand((B, L), generator=g) * 10.0
    # a slowly falling profile with noise, so the prefix minima fall in steps
    s = s + torch.linspace(20, 0, L)[None, :]
    return s.float()


@pytest.mark.parametrize("L", [1, 7, 1000, 1025, 4096, 70001])
@pytest.mark.parametrize("lo,hi", [(0.0, 1.0), (0.1, 0.25), (0.3, 0.3), (1.0, 1.0)])
def test_adaptive_prefix_matches_oracle(dl, L, lo, hi):
    g = torch.Generator().manual_seed(L)
    B = 5
    s = _scores(g, B, L)
    start = torch.tensor([0, L // 3, max(L - 1, 0), L, L // 2], dtype=torch.int32)
    length, tau = dl.dllm_adaptive_prefix(s.cuda(), start.cuda(), lo, hi)
    torch.cuda.synchronize()
    ref_len, ref_tau = oracle.adaptive_prefix(s.numpy(), start.numpy(), lo, hi)
    assert np.array_equal(length.cpu().numpy(), ref_len)
    assert np.array_equal(tau.cpu().numpy(), ref_tau)


def test_adaptive_prefix_special_values_and_advance(dl):
    g = torch.Generator().manual_seed(3)
    B, L = 6, 3000
    s = _scores(g, B, L)
    s[0, 17] = float("nan")           # NaN inside the lower fraction: tau -inf, stop there
    s[1, 2500] = float("nan")         # NaN past it
    s[2, :] = float("inf")            # all committed: tau +inf, length capped at hi A
    s[3, 100:] = -float("inf")
    s[4, 0] = float("nan")            # NaN first: fallback of one token
    start = torch.tensor([0, 0, 0, 50, 0, 2990], dtype=torch.int32)
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    start_d = start.cuda()
    length, tau = dl.dllm_adaptive_prefix(s.cuda(), start_d, 0.05, 0.5, advance_start=True,
                                          dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    ref_len, ref_tau = oracle.adaptive_prefix(s.numpy(), start.numpy(), 0.05, 0.5)
    assert np.array_equal(length.cpu().numpy(), ref_len)
    assert np.array_equal(tau.cpu().numpy(), ref_tau)
    assert np.array_equal(start_d.cpu().numpy(), start.numpy() + ref_len)
    assert ref_len[4] == 1 and ref_len[0] == 17


def test_adaptive_prefix_bad_start_reports(dl):
    s = torch.zeros((2, 10), device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    length, _ = dl.dllm_adaptive_prefix(s, torch.tensor([3, 11], dtype=torch.int32, device="cuda"),
                                        0.1, 0.5, dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) != 0 and int(length[1]) == 0


# ------------------------------------------------ criterion with the confidence

CONF_RTOL = 1e-4  # float32 sum of up to 126464 exponentials, as for dllm_confidence


def _check_conf(conf, am, mg, rc, ra, rm, mask):
    assert np.array_equal(i32_(am)[mask], ra[mask])
    g, r = f64(conf)[mask], rc[mask]
    assert np.all(np.abs(g - r) <= 1e-6 + CONF_RTOL * np.abs(r)), np.max(np.abs(g - r) / r)
    assert np.max(np.abs(f64(mg)[mask] - rm[mask]), initial=0.0) <= 1e-6


def i32_(t):
    return t.detach().cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("dtype,V,B", [(torch.float32, 301, 3), (torch.bfloat16, 1000, 3),
                                       (torch.bfloat16, 126464, 3), (torch.bfloat16, 1000, 65),
                                       (torch.float32, 4096, 65)])
def test_lock_conf_matches_oracle(dl, dtype, V, B):
    """dllm_lock_criterion_conf: the divergences and uncertainties of the
    criterion and the confidence, argmax and margin of the current rows, with
    ragged counts (persistent partial kernel at 3 batch rows, one CTA per row
    slot at 65), against the oracle's lock_kl and confidence."""
    g = torch.Generator().manual_seed(V + B)
    R = 9
    z, y = _pair(g, B, R, V, dtype, 1.0)
    count = torch.tensor([(5 * b + 3) % (R + 1) for b in range(B)], dtype=torch.int32)
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    kl, unc, _, conf, am, mg = dl.dllm_lock_criterion_conf(z.cuda(), y.cuda(), 0.0,
                                                           count=count.cuda(), dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    mask = np.arange(R)[None, :] < count.numpy()[:, None]
    ref_kl, ref_unc = oracle.lock_kl(f64(z), f64(y))
    _check_kl(kl, unc, ref_kl, ref_unc, mask)
    rc, ra, rm = oracle.confidence(f64(z))
    _check_conf(conf, am, mg, rc, ra, rm, mask)
    # the uncertainty is the complement of the confidence, before its clamp at 0
    assert np.array_equal(f64(unc)[mask], np.maximum(1.0 - f64(conf)[mask].astype(np.float32), 0))


def test_lock_conf_ties_gather_scatter_flags(dl):
    """Ties for the maximum inside one chunk and across chunks (argmax the
    lowest index, margin 0), rows gathered by index and results scattered to
    positions, lock flags, and the same outputs as dllm_confidence and
    dllm_lock_criterion called separately on the same rows."""
    g = torch.Generator().manual_seed(23)
    B, R_src, V, L, R_max = 2, 12, 126464, 64, 8
    z, y = _pair(g, B, R_src, V, torch.bfloat16, 2.0)
    top = float(z.float().max()) + 1.0
    z[0, 0, 5] = z[0, 0, 7] = top          # tie inside the first chunk
    z[0, 1, 100] = z[0, 1, 120000] = top   # tie across chunks: the lower index wins
    z[1, 2, V - 1] = top                   # maximum on the last element of the row
    count = torch.tensor([8, 5], dtype=torch.int32)
    row_idx = torch.stack([torch.arange(R_max), torch.arange(R_max) + 2]).int()
    out_idx = torch.stack([torch.randperm(L, generator=g)[:R_max] for _ in range(B)]).int()
    args = dict(gate_q=0.5, R_max=R_max, row_idx=row_idx.cuda(), count=count.cuda(),
                out_idx=out_idx.cuda(), out_cols=L)
    lk1 = torch.zeros((B, L), dtype=torch.uint8, device="cuda")
    lk2 = lk1.clone()
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    zc, yc = z.cuda(), y.cuda()
    kl, unc, _, conf, am, mg = dl.dllm_lock_criterion_conf(
        zc, yc, 1e-2, locked_inout=lk1, conf_out=torch.full((B, L), -7.0, device="cuda"),
        dev_status=st, **args)
    kl2, unc2, _ = dl.dllm_lock_criterion(zc, yc, 1e-2, locked_inout=lk2, dev_status=st, **args)
    conf2, am2, mg2 = dl.dllm_confidence(zc, R_max=R_max, row_idx=row_idx.cuda(),
                                         count=count.cuda(), out_idx=out_idx.cuda(), out_cols=L,
                                         dev_status=st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    rc, ra, rm = oracle.confidence(f64(z), count=count.numpy(), row_idx=row_idx.numpy())
    for b in range(B):
        n = int(count[b])
        cols = out_idx[b, :n].numpy()
        m = np.ones(n, dtype=bool)
        _check_conf(conf[b:b + 1, cols], am[b:b + 1, cols], mg[b:b + 1, cols],
                    rc[b:b + 1, :n], ra[b:b + 1, :n], rm[b:b + 1, :n], m[None, :])
        # against the two separate calls: the same criterion, argmax and margin
        assert np.array_equal(f64(kl)[b, cols], f64(kl2)[b, cols])
        assert np.array_equal(f64(unc)[b, cols], f64(unc2)[b, cols])
        assert np.array_equal(i32_(am)[b, cols], i32_(am2)[b, cols])
        assert np.array_equal(f64(mg)[b, cols], f64(mg2)[b, cols])
        gc, sc = f64(conf)[b, cols], f64(conf2)[b, cols]
        assert np.all(np.abs(gc - sc) <= 2 * CONF_RTOL * sc)
        # columns of no row keep their values
        rest = np.setdiff1d(np.arange(L), cols)
        assert np.all(f64(conf)[b, rest] == -7.0)
    assert i32_(am)[0, out_idx[0, 0]] == 5 and f64(mg)[0, out_idx[0, 0]] == 0.0
    assert i32_(am)[0, out_idx[0, 1]] == 100 and f64(mg)[0, out_idx[0, 1]] == 0.0
    assert i32_(am)[1, out_idx[1, 0]] == V - 1
    assert torch.equal(lk1, lk2)
