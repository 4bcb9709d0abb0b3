"""Plain float64 definitions of every output of the partial denoising step.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path.

Inputs are numpy arrays already decoded to float64 (decoding a bfloat16 or
float32 value to float64 is exact).  Nothing here is blocked, fused or
reordered: each function evaluates the definition it cites, with numpy's
matmul / sum / exp / argmax as the only library steps.

Pages cited (title, then section):

* DyLLM -- "DyLLM: Efficient Diffusion LLM Inference via Saliency-based Token
  Selection and Partial Attention".
* SlowFast -- "Accelerating Diffusion Large Language Models with SlowFast
  Sampling: The Three Golden Principles".
* Attn-Sampler -- "Attention-Based Sampler for Diffusion Language Models".
* SureLock -- "Stopping Computation for Converged Tokens in Masked
  Diffusion-LM Decoding".
* LSP -- "Beyond Scattered Acceptance: Fast and Coherent Inference for DLMs via
  Longest Stable Prefixes".

Readings taken where the pages are silent (each is pinned or listed as
unpinned in the tests): salient iff cos < tau, so cos == tau is stable and a
NaN cosine is salient; two zero vectors have cosine 1, one zero vector gives 0;
compaction keeps ascending positions and pads with -1; confidence is the
maximum of a temperature-1 softmax; argmax ties go to the lowest vocabulary
index and then the margin is 0; attention is unmasked (bidirectional) with
scale 1/sqrt(d); column sums add the row-normalised probabilities of the
active query rows only; a prefix position is stable iff score >= tau, NaN is
unstable.  Around the step: the lock criterion's percentile is taken over the
active rows of a batch row; the adaptive prefix threshold is the prefix
minimum at the lower end of the fraction range; the stable rows' existing
attention weights are the previous step's, recovered from the cached query,
keys and log-sum-exp; the decoding order's dynamic threshold is
max(tau, gamma * top score); structural boundaries are caller-given flags per
vocabulary id; the SlowFast convergence point is tracked by the exact
population variance of a window of predictions; the fast phase unmasks the
masked tokens of [start, region end) with confidence strictly above the
high threshold, the slow phase the k most confident masked tokens of the
exploration window [start, start + width).  Each function's docstring
states its reading in full.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

__all__ = [
    "saliency_cos",
    "salient_flags",
    "compact",
    "saliency_select",
    "confidence",
    "kv_scatter",
    "partial_attention",
    "stable_prefix",
    "lock_kl",
    "lock_decision",
    "adaptive_prefix",
    "approx_attention_update",
    "attn_scores",
    "attn_sampler_select",
    "slowfast_phases",
    "slowfast_fast_select",
    "slowfast_slow_select",
    "slowfast_select",
    "snap_prefix",
    "step",
]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# Saliency: temporal cosine similarity, threshold, ordered compaction
# --------------------------------------------------------------------------

def saliency_cos(cur, prev) -> np.ndarray:
    """Temporal cosine similarity of each position's current and cached vector.

    DyLLM, technical summary, Methodology 1 (layer-adaptive saliency
    selection), "Meting": s_{t,l} is the cosine similarity, per token and per
    layer, of the vector at step t and the cached one from step t-1.

    ``cur``/``prev``: [..., D].  Returns cos [...] in float64.  Both vectors
    zero -> 1 (identical); exactly one zero -> 0.
    """
    cur = _f64(cur)
    prev = _f64(prev)
    dot = np.sum(cur * prev, axis=-1)
    n_cur = np.sqrt(np.sum(cur * cur, axis=-1))
    n_prev = np.sqrt(np.sum(prev * prev, axis=-1))
    out = np.empty(dot.shape, dtype=np.float64)
    both_zero = (n_cur == 0.0) & (n_prev == 0.0)
    one_zero = (n_cur == 0.0) != (n_prev == 0.0)
    regular = ~(both_zero | one_zero)
    out[regular] = dot[regular] / (n_cur[regular] * n_prev[regular])
    out[both_zero] = 1.0
    out[one_zero] = 0.0
    return out


def salient_flags(cos, tau: float, locked=None) -> np.ndarray:
    """Active = salient and not locked.

    DyLLM, technical summary, Methodology 1, "Selectie": a cosine close to 1 is
    stable, a low cosine is salient and is recomputed (tau = 0.99 in the
    results).  SureLock, technical summary section 2 ("Berechnungsoptimierung"):
    locked positions skip their own recompute.

    The comparison is taken in float32, the precision the kernel stores its
    cosine in: salient iff float32(cos) < float32(tau), NaN salient.
    """
    c32 = np.asarray(cos).astype(np.float32)
    t32 = np.float32(tau)
    active = ~(c32 >= t32)
    if locked is not None:
        active &= ~np.asarray(locked).astype(bool)
    return active


def compact(flags, idx_base: int = 0):
    """Ordered stream compaction of the active flags of each batch row.

    DyLLM, technical summary, Methodology 1, "Optimalisatie": only the salient
    rows are recomputed, the rest reuse the cache -- so the recompute needs the
    list of salient positions.  Returns idx [B, Lw] int32 (ascending positions
    + ``idx_base``, padded with -1) and count [B] int32.
    """
    flags = np.asarray(flags, dtype=bool)
    B, Lw = flags.shape
    idx = np.full((B, Lw), -1, dtype=np.int32)
    count = np.zeros(B, dtype=np.int32)
    for b in range(B):
        pos = np.flatnonzero(flags[b])
        idx[b, : len(pos)] = pos + idx_base
        count[b] = len(pos)
    return idx, count


def saliency_select(cur, prev, tau: float, locked=None, idx_base: int = 0):
    """Cosine, threshold and compaction over a [B, Lw, D] window.

    DyLLM, technical summary, Methodology 1 (measurement, selection) and 3
    (adaptive input: the window is the response rows on most steps and the
    whole sequence every few steps).  Returns (cos [B, Lw] float64,
    idx [B, Lw] int32, count [B] int32).
    """
    cos = saliency_cos(cur, prev)
    idx, count = compact(salient_flags(cos, tau, locked), idx_base)
    return cos, idx, count


# --------------------------------------------------------------------------
# Confidence, argmax and logit margin over the vocabulary
# --------------------------------------------------------------------------

def confidence(logits, count=None, row_idx=None):
    """Max softmax probability, argmax and top-1 minus top-2 logit per row.

    SlowFast, section 2 (certainty principle; fast phase unmasks tokens whose
    confidence exceeds a high threshold); SureLock, technical summary section 2,
    locking criterion 2 (uncertainty 1 - max_v p(v)); LSP, technical summary
    section 2, step 1 (logit margin = highest minus second-highest logit).

    ``logits``: [B, R, V].  Row r of batch b reads ``logits[b, row_idx[b, r]]``
    when ``row_idx`` ([B, R_max]) is given, else ``logits[b, r]``; rows
    r >= count[b] are skipped (NaN / -1).  Returns conf, argmax, margin, each
    [B, R_max].
    """
    z_all = _f64(logits)
    B, R, V = z_all.shape
    R_max = R if row_idx is None else np.asarray(row_idx).shape[1]
    if count is None:
        count = np.full(B, R_max, dtype=np.int64)
    conf = np.full((B, R_max), np.nan)
    amax = np.full((B, R_max), -1, dtype=np.int32)
    margin = np.full((B, R_max), np.nan)
    for b in range(B):
        for r in range(int(count[b])):
            row = r if row_idx is None else int(row_idx[b][r])
            z = z_all[b, row]
            j = int(np.argmax(z))  # first occurrence: lowest index on ties
            m = z[j]
            conf[b, r] = 1.0 / np.sum(np.exp(z - m))
            amax[b, r] = j
            rest = np.concatenate([z[:j], z[j + 1:]])
            margin[b, r] = m - np.max(rest)
    return conf, amax, margin


# --------------------------------------------------------------------------
# KV cache update
# --------------------------------------------------------------------------

def kv_scatter(k_cache, v_cache, k_new, v_new, idx, count):
    """Write the fresh K/V rows of the active positions into the full cache.

    SureLock, technical summary section 2: K/V of locked positions are cached
    and other tokens keep attending to them; only active rows get new K/V.
    LSP, technical summary section 2 ("KV Cache"): contiguous appends.

    Caches [B, L, H, d]; new rows [B, M_max, H, d]; row i < count[b] goes to
    position idx[b, i].  Returns updated copies (inputs are left alone).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    for b in range(kc.shape[0]):
        for i in range(int(count[b])):
            p = int(idx[b][i])
            kc[b, p] = k_new[b, i]
            vc[b, p] = v_new[b, i]
    return kc, vc


# --------------------------------------------------------------------------
# Partial attention and attention column sums
# --------------------------------------------------------------------------

def partial_attention(q, k_cache, v_cache, count, scale: Optional[float] = None):
    """Exact softmax attention of the active query rows over every cached key.

    DyLLM, technical summary, Methodology 2 (salient path: the score rows of
    salient queries are recomputed in full); SureLock, technical summary
    section 2 (active tokens attend to all positions through the cached K/V;
    cost O(M N d)); Attn-Sampler, technical summary, Methodology 2 (column sums
    of the attention matrix).

    q [B, M_max, H, d] (rows i < count[b] are the active queries), caches
    [B, L, H, d].  Per (b, h): S = scale * Q K^T (no mask: the models are
    bidirectional), P = row softmax of S, O = P V, lse = log sum_j exp S,
    colsum[j] = sum over active rows of P[:, j].  Returns o [B, M_max, H, d]
    (NaN on inactive rows), lse [B, H, M_max] (NaN on inactive rows),
    colsum [B, H, L].
    """
    q = _f64(q)
    k = _f64(k_cache)
    v = _f64(v_cache)
    B, M_max, H, d = q.shape
    L = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.full((B, M_max, H, d), np.nan)
    lse = np.full((B, H, M_max), np.nan)
    colsum = np.zeros((B, H, L))
    for b in range(B):
        n = int(count[b])
        if n == 0:
            continue
        for h in range(H):
            Q = q[b, :n, h, :]
            K = k[b, :, h, :]
            Vv = v[b, :, h, :]
            S = scale * (Q @ K.T)
            m = np.max(S, axis=1, keepdims=True)
            E = np.exp(S - m)
            l = np.sum(E, axis=1, keepdims=True)
            P = E / l
            o[b, :n, h, :] = P @ Vv
            lse[b, h, :n] = (m + np.log(l))[:, 0]
            colsum[b, h, :] = np.sum(P, axis=0)
    return o, lse, colsum


# --------------------------------------------------------------------------
# Longest stable prefix
# --------------------------------------------------------------------------

def stable_prefix(score, start, tau: float, min_commit: bool = True):
    """Length of the longest run of stable positions starting at ``start``.

    LSP, technical summary section 2: commit the longest contiguous stable
    block at the head of the remaining active suffix (core principle), using a
    per-position stability score (step 1); step 4 (fallback) commits at least
    one token when none is stable.

    ``score`` [B, L]; stable iff float32(score) >= float32(tau) (NaN is not).
    Returns len [B] int32.
    """
    s32 = np.asarray(score).astype(np.float32)
    t32 = np.float32(tau)
    B, L = s32.shape
    out = np.zeros(B, dtype=np.int32)
    for b in range(B):
        st = int(start[b])
        k = 0
        while st + k < L and s32[b, st + k] >= t32:
            k += 1
        if min_commit and k == 0 and st < L:
            k = 1
        out[b] = k
    return out


# --------------------------------------------------------------------------
# Lock criterion (SureLock) and adaptive prefix threshold (LSP)
# --------------------------------------------------------------------------

def lock_kl(logits_cur, logits_prev, count=None, row_idx=None):
    """Local KL divergence between consecutive steps and the uncertainty.

    SureLock, technical summary section 2, locking criterion 1: the local
    divergence D = KL(p_t || p_{t-1}) between the current and the previous
    step's predictive distribution of a position; criterion 2: its
    uncertainty 1 - max_v p_t(v).

    ``logits_cur``/``logits_prev`` [B, R, V] (same row layout); row r of batch
    b reads row ``row_idx[b, r]`` when given, else row r; rows r >= count[b]
    are skipped (NaN).  p = softmax(z), q = softmax(y), and with the
    log-softmax log p_j = z_j - logsumexp(z):
    KL = sum_j p_j (log p_j - log q_j).  Returns kl, unc, each [B, R_max].
    """
    z_all, y_all = _f64(logits_cur), _f64(logits_prev)
    B, R, V = z_all.shape
    R_max = R if row_idx is None else np.asarray(row_idx).shape[1]
    if count is None:
        count = np.full(B, R_max, dtype=np.int64)
    kl = np.full((B, R_max), np.nan)
    unc = np.full((B, R_max), np.nan)
    for b in range(B):
        for r in range(int(count[b])):
            row = r if row_idx is None else int(row_idx[b][r])
            z, y = z_all[b, row], y_all[b, row]
            mz, my = np.max(z), np.max(y)
            log_p = z - (mz + np.log(np.sum(np.exp(z - mz))))
            log_q = y - (my + np.log(np.sum(np.exp(y - my))))
            p = np.exp(log_p)
            kl[b, r] = np.sum(p * (log_p - log_q))
            unc[b, r] = 1.0 - np.max(p)
    return kl, unc


def lock_decision(kl, unc, count, eps: float, gate_q: float):
    """Which active rows lock at this step.

    SureLock, technical summary section 2: a position locks when its local
    KL divergence is below eps (criterion 1) and, with the optional gate
    (criterion 2), its uncertainty lies below a percentile of the
    uncertainties.  Reading: the percentile is taken over the active rows of
    the same batch row; with n of them and gate fraction q in (0, 1), the gate
    passes iff unc <= the k-th smallest uncertainty, k = max(1, ceil(q n));
    q <= 0 or q >= 1 disables the gate; q is taken as a float32 and q n is
    the exact product.  Decisions compare float32 values (kl < eps, unc <=
    threshold); NaN never locks.  Returns lock [B, R_max]
    (bool).
    """
    kl32 = np.asarray(kl, dtype=np.float32)
    unc32 = np.asarray(unc, dtype=np.float32)
    B, R_max = kl32.shape
    lock = np.zeros((B, R_max), dtype=bool)
    for b in range(B):
        n = int(count[b])
        if n == 0:
            continue
        gate = np.ones(n, dtype=bool)
        if 0.0 < gate_q < 1.0:
            u = unc32[b, :n]
            k = max(1, int(math.ceil(float(np.float32(gate_q)) * n)))
            finite = np.sort(u[~np.isnan(u)])
            t = finite[k - 1] if k <= len(finite) else np.float32(np.inf)
            gate = u <= t
        lock[b, :n] = (kl32[b, :n] < np.float32(eps)) & gate
    return lock


def adaptive_prefix(score, start, lo: float, hi: float):
    """Longest stable prefix with an adaptive threshold.

    LSP, technical summary section 2, step 2 (adaptive sizing): instead of a
    fixed threshold, tau is chosen so that the committed stable block covers
    a fraction [lo, hi] of the current active length A = L - start; step 4
    (fallback): at least one token.  Reading: with the prefix minima
    m_k = min(score[start .. start + k - 1]) (NaN counts as unstable, -inf),
    k_lo = max(1, ceil(lo A)) and k_hi = max(k_lo, floor(hi A)) (lo, hi taken
    as float32, the products exact):
    tau = m_{k_lo}, len = min(k_hi, #{k : m_k >= tau}), never past the first
    NaN score, and at least 1 when A > 0.  Scores are compared as float32.
    Returns (len [B] int32, tau [B] float32; +inf when A = 0).
    """
    s32 = np.asarray(score).astype(np.float32)
    B, L = s32.shape
    lens = np.zeros(B, dtype=np.int32)
    taus = np.full(B, np.inf, dtype=np.float32)
    for b in range(B):
        st = int(start[b])
        A = L - st
        if A <= 0:
            continue
        seg = s32[b, st:]
        m = np.empty(A, dtype=np.float32)
        cur = np.float32(np.inf)
        first_nan = A
        for k in range(A):
            v = seg[k]
            if np.isnan(v):
                v = np.float32(-np.inf)
                first_nan = min(first_nan, k)
            cur = min(cur, v)
            m[k] = cur
        k_lo = max(1, int(math.ceil(float(np.float32(lo)) * A)))
        k_lo = min(k_lo, A)
        k_hi = max(k_lo, int(math.floor(float(np.float32(hi)) * A)))
        tau = m[k_lo - 1]
        n_ge = 0
        while n_ge < A and m[n_ge] >= tau:
            n_ge += 1
        ln = min(k_hi, n_ge, first_nan)
        lens[b] = max(ln, 1)
        taus[b] = tau
    return lens, taus


# --------------------------------------------------------------------------
# Approximate attention update of the stable rows (the non-salient path)
# --------------------------------------------------------------------------

def approx_attention_update(o_prev, q_prev, lse_prev, k_prev, v_prev, v_new, idx, count,
                            stable_idx, stable_count, scale: Optional[float] = None):
    """Output of the stable rows after this step's value changes.

    DyLLM, technical summary, Methodology 2 (non-salient path): for a stable
    row the change of its attention weights is taken as negligible, and its
    output is updated by the change of the value vectors of the salient
    tokens weighted by the existing attention weights; cost O(N |A_t|).
    Reading: the existing weights are the previous step's softmax row,
    recovered exactly from the cached query, the previous keys of the salient
    positions and the cached log-sum-exp:
    p_ij = exp(scale q_i . k_j - lse_i), and
    o_i <- o_i + sum_{a < count} p_{i, idx_a} (v_new_a - v_prev[idx_a]).

    o_prev, q_prev, k_prev, v_prev [B, L, H, d] (the previous step's outputs,
    queries, keys and values of every position; k_prev and v_prev before this
    step's cache update); lse_prev [B, H, L]; v_new [B, M_max, H, d], row a
    the fresh value of position idx[b, a] for a < count[b]; stable rows
    stable_idx[b, r] for r < stable_count[b].  Returns an updated copy of
    o_prev (only the stable rows change).
    """
    o = np.array(_f64(o_prev), copy=True)
    q, lse, k, v, vn = (_f64(x) for x in (q_prev, lse_prev, k_prev, v_prev, v_new))
    B, L, H, d = o.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for b in range(B):
        A = [int(idx[b][a]) for a in range(int(count[b]))]
        rows = [int(stable_idx[b][r]) for r in range(int(stable_count[b]))]
        if not A or not rows:
            continue
        for h in range(H):
            Q = q[b, rows, h, :]                       # [N, d]
            K_A = k[b, A, h, :]                        # [|A|, d]
            dV = vn[b, :len(A), h, :] - v[b, A, h, :]  # [|A|, d]
            P = np.exp(scale * (Q @ K_A.T) - lse[b, h, rows][:, None])
            o[b, rows, h, :] += P @ dV
    return o


# --------------------------------------------------------------------------
# Attention-guided decoding order (Attn-Sampler)
# --------------------------------------------------------------------------

def attn_scores(colsum):
    """Total attention each position receives.

    Attn-Sampler, technical summary, Methodology 1 (key insight: decode in
    descending order of the column sums of the attention matrix) and the
    ablation on layers and heads (aggregating over all of them works best).
    colsum [B, ..., L] (per head, or per layer and head); returns the sum over
    every axis between the batch and the position axis, [B, L].
    """
    c = _f64(colsum)
    return c.reshape(c.shape[0], -1, c.shape[-1]).sum(axis=1)


def attn_sampler_select(score, candidates, tau: float, gamma: float, k_max: int):
    """Decoding order and the number of tokens to decode in parallel.

    Attn-Sampler, technical summary, Methodology 2: tokens with the highest
    column sums are decoded first (order determination); tokens are decoded
    in parallel only while their score exceeds a threshold (parallel
    decoding).  The page does not print the dynamic threshold; reading: the
    threshold of a step is thr = max(tau, gamma * a_top), a floor given by the
    caller and a fraction of that step's top score (gamma = 1 gives one token
    per step unless the top is tied; gamma <= 0 drops the second term, a
    static threshold).

    score [B, L] (compared as float32); candidates [B, L] nonzero where a
    position may be decoded (None: all).  order[b] lists the candidates by
    descending score, equal scores by ascending position, NaN last (-0 and +0
    are equal), padded with -1; n[b] is the number of leading entries with
    score >= thr (float32, thr = max(float32 tau, float32(gamma) * a_top
    rounded to float32) for gamma > 0, else float32 tau), capped at k_max
    when k_max > 0, and at least 1 when there is a candidate.  Returns order [B, L] int32, n [B] int32.
    """
    s32 = np.asarray(score, dtype=np.float32)
    B, L = s32.shape
    order = np.full((B, L), -1, dtype=np.int32)
    n_out = np.zeros(B, dtype=np.int32)
    for b in range(B):
        cand = [j for j in range(L) if candidates is None or candidates[b][j]]
        if not cand:
            continue

        def key(j):
            v = float(s32[b, j])
            return (1, 0.0, j) if math.isnan(v) else (0, -v, j)

        ranked = sorted(cand, key=key)
        order[b, :len(ranked)] = ranked
        top = s32[b, ranked[0]]
        thr = np.float32(tau)
        if gamma > 0:
            thr = max(thr, np.float32(np.float32(gamma) * top))
        n = 0
        while n < len(ranked) and s32[b, ranked[n]] >= thr:
            n += 1
        if k_max > 0:
            n = min(n, k_max)
        n_out[b] = max(n, 1)
    return order, n_out


# --------------------------------------------------------------------------
# Structural snapping of the committed block
# --------------------------------------------------------------------------

def snap_prefix(tokens, delim, start, length, min_len: int):
    """Length of the committed block after structural snapping.

    LSP, technical summary section 2, step 3 (structural snapping): the end
    of the selected block is moved to the nearest natural boundary
    (punctuation, newline, code symbol) inside the candidate block, so that
    no word or sentence is frozen half way.  Reading: the tokenizer's
    delimiter set is given as a flag per vocabulary id; the block
    [start, start + length) ends after its last delimiter token at a position
    p >= start + max(min_len, 1) - 1, i.e. the new length is p - start + 1;
    with no such delimiter the length is unchanged.

    tokens [B, L] (e.g. the argmax of each position), delim [V], start and
    length [B].  Returns the snapped lengths [B] int32.
    """
    tok = np.asarray(tokens)
    out = np.array(length, dtype=np.int32, copy=True)
    for b in range(tok.shape[0]):
        s, n = int(start[b]), int(length[b])
        lo = s + max(int(min_len), 1) - 1
        for p in range(s + n - 1, lo - 1, -1):
            if delim[int(tok[b, p])]:
                out[b] = p - s + 1
                break
    return out


# --------------------------------------------------------------------------
# SlowFast phase control
# --------------------------------------------------------------------------

def slowfast_phases(starts, e_cands, window: int, sigma2: float):
    """Phase and region of each step of SlowFast sampling.

    SlowFast, section 2 (pipeline): in the slow (exploratory) phase the
    prediction of the convergence point e_cand is watched over a sliding
    window of steps; when the variance of the prediction falls below
    sigma^2_stable the region [s_cycle, e_cycle] is stable and the fast phase
    decodes it in one step; then a new cycle starts.  Reading: one cycle
    starts empty; each step appends that step's e_cand; with the last
    ``window`` predictions x_1 .. x_W of the cycle, the region is stable iff
    their population variance is below sigma2 (evaluated exactly as
    W sum x^2 - (sum x)^2 < sigma2 W^2, the right side in float64) and the
    latest prediction lies beyond the start; that step is fast with region
    [start, latest e_cand), and the next step begins a new cycle.

    starts, e_cands: [T, B] integers (start of the undecoded suffix and the
    prediction at each step).  Returns phase [T, B] (0 slow, 1 fast) and
    region end [T, B] (the region's end on fast steps, -1 otherwise).
    """
    T, B = len(starts), len(starts[0])
    phase = np.zeros((T, B), dtype=np.int32)
    end = np.full((T, B), -1, dtype=np.int32)
    for b in range(B):
        hist = []
        for t in range(T):
            hist.append(int(e_cands[t][b]))
            if len(hist) > window:
                hist.pop(0)
            if len(hist) == window and hist[-1] > int(starts[t][b]):
                num = window * sum(x * x for x in hist) - sum(hist) ** 2
                if num < float(sigma2) * (window * window):
                    phase[t, b] = 1
                    end[t, b] = hist[-1]
                    hist = []
    return phase, end


def slowfast_fast_select(conf, masked, start, region_end, tau_high: float):
    """Tokens the fast phase unmasks in one step.

    SlowFast, section 2 (pipeline, accelerated decoding phase): once the
    region [s_cycle, e_cycle] is stable, every still-masked token of the
    region whose confidence exceeds the high threshold tau_high_conf is
    unmasked at the same time.  Reading: the region is [start, region_end)
    (the controller's region: from the start of the undecoded suffix to the
    latest convergence prediction); "exceeds" is strict, conf > tau_high,
    compared in float32 (NaN never passes); no fallback -- a region with no
    such token unmasks nothing.

    conf [B, L] (e.g. the confidence of dllm_confidence), masked [B, L]
    nonzero where a position is still masked (None: all), start and
    region_end [B].  Returns idx [B, L] int32 (ascending positions, -1 pad)
    and count [B] int32.
    """
    c32 = np.asarray(conf, dtype=np.float32)
    B, L = c32.shape
    t32 = np.float32(tau_high)
    idx = np.full((B, L), -1, dtype=np.int32)
    count = np.zeros(B, dtype=np.int32)
    for b in range(B):
        lo, hi = max(int(start[b]), 0), min(int(region_end[b]), L)
        sel = [p for p in range(lo, hi)
               if (masked is None or masked[b][p]) and c32[b, p] > t32]
        idx[b, :len(sel)] = sel
        count[b] = len(sel)
    return idx, count


def slowfast_slow_select(conf, masked, start, width: int, k: int):
    """Tokens the slow (exploratory) phase unmasks in one step.

    SlowFast, section 2 (pipeline, exploratory phase): the model decodes
    cautiously, selecting the tokens with the highest confidence in an
    exploration window.  Reading: the window is [start, start + width) cut at
    L; its still-masked positions with a non-NaN confidence are ranked by
    descending float32 confidence, equal confidences by ascending position;
    the first min(k, candidates) are selected.  Returned in ascending
    position order: idx [B, L] int32 (-1 pad), count [B] int32.
    """
    c32 = np.asarray(conf, dtype=np.float32)
    B, L = c32.shape
    idx = np.full((B, L), -1, dtype=np.int32)
    count = np.zeros(B, dtype=np.int32)
    for b in range(B):
        lo = max(int(start[b]), 0)
        hi = min(lo + int(width), L)
        cand = [p for p in range(lo, hi)
                if (masked is None or masked[b][p]) and not np.isnan(c32[b, p])]
        ranked = sorted(cand, key=lambda p: (-float(c32[b, p]), p))
        sel = sorted(ranked[:max(int(k), 0)])
        idx[b, :len(sel)] = sel
        count[b] = len(sel)
    return idx, count


def slowfast_select(conf, masked, start, phase, region_end, tau_high: float, width: int, k: int):
    """One SlowFast step's unmasked tokens, per batch row: the fast phase's
    (phase 1, region [start, region_end)) or the slow phase's (phase 0)."""
    B = len(start)
    fi, fc = slowfast_fast_select(conf, masked, start, region_end, tau_high)
    si, sc = slowfast_slow_select(conf, masked, start, width, k)
    idx = np.where(np.asarray(phase)[:, None] == 1, fi, si).astype(np.int32)
    count = np.where(np.asarray(phase) == 1, fc, sc).astype(np.int32)
    assert idx.shape[0] == B
    return idx, count


# --------------------------------------------------------------------------
# One whole partial step
# --------------------------------------------------------------------------

def step(cur, prev, k_cache, v_cache, k_new, v_new, q, logits, *, tau: float,
         win_start: int, score, start, tau_c: float, min_commit: bool = True,
         scale: Optional[float] = None, locked=None):
    """One partial denoising step, composed in the order the pages give.

    Select the salient rows of the window (DyLLM), write their fresh K/V into
    the cache (SureLock), attend from them over the whole cache with column
    sums (DyLLM, Attn-Sampler), score the window's logit rows (SlowFast,
    SureLock, LSP) and find the committable prefix (LSP).  ``logits`` holds one
    row per window position; their confidence replaces ``score`` there.
    """
    cos, idx, count = saliency_select(cur[:, win_start:], prev[:, win_start:], tau,
                                      locked, idx_base=win_start)
    kc, vc = kv_scatter(k_cache, v_cache, k_new, v_new, idx, count)
    o, lse, colsum = partial_attention(q, kc, vc, count, scale)
    conf, amax, margin = confidence(logits)
    new_score = np.array(score, dtype=np.float64, copy=True)
    R = conf.shape[1]
    new_score[:, win_start:win_start + R] = conf
    length = stable_prefix(new_score, start, tau_c, min_commit)
    return dict(cos=cos, idx=idx, count=count, k_cache=kc, v_cache=vc, o=o,
                lse=lse, colsum=colsum, conf=conf, argmax=amax, margin=margin,
                score=new_score, length=length)
