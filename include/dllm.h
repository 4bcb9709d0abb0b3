/*
 * dllm.h -- C ABI of the partial denoising step for masked-diffusion language
 * models (one step that recomputes only a selected subset of token positions).
 *
 * The library (libdllm.so) runs every entry point as CUDA kernels for sm_103a
 * (B300) on the caller's stream (the SlowFast controller is plain host code).
 * It never allocates device memory, never synchronises the stream and never
 * reads device data back to the host: the active-row counts stay on the
 * device, so a whole step can be captured in a CUDA graph.
 *
 * Entry points
 *   The step, in order: dllm_saliency_select, dllm_kv_scatter,
 *   dllm_partial_attention (with or without column sums; the sums alone:
 *   dllm_attention_colsum), dllm_confidence (dllm_confidence_static_ws for
 *   callers that cannot allocate), dllm_stable_prefix.
 *   Around it: dllm_lock_criterion (SureLock; dllm_lock_criterion_conf also
 *   gives dllm_confidence's outputs), dllm_adaptive_prefix and
 *   dllm_snap_prefix (LSP), dllm_approx_attention_update (DyLLM's stable
 *   rows), dllm_attn_scores and dllm_attn_sampler_select (Attn-Sampler), and
 *   the host-side SlowFast controller dllm_slowfast_create / _observe /
 *   _destroy, its device twin dllm_slowfast_observe_device and the tokens
 *   each SlowFast phase unmasks, dllm_slowfast_select.
 *
 * Common conventions
 *   - Every data pointer is a DEVICE pointer owned by the caller (the SlowFast
 *     controller's arrays excepted: host memory).  Inputs are read only;
 *     outputs are written only where stated.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Element types: DLLM_F32 (IEEE float32) or DLLM_BF16 (bfloat16).  Scores,
 *     log-sum-exps and column sums are always float32; indices int32.
 *   - Sizes given on the host (M_max, R_max, ...) size the launch; the actual
 *     per-batch counts are read on the device.
 *   - Host-side validation failures return before any launch.  A failed launch
 *     returns DLLM_ERR_CUDA.  dllm_last_error() then describes the failure
 *     (thread-local string, valid until the next failing call on the thread).
 *   - `dev_status` (may be NULL): an int32 in device memory that the caller
 *     zeroes.  A kernel that detects bad device-side data (a count outside
 *     [0, M_max], an index out of range or out of order, a bounded wait that
 *     ran out) stores the first such code there (DLLM_ERR_DEVICE_CHECK or
 *     DLLM_ERR_TIMEOUT), skips the offending row and carries on; it never
 *     traps.  The caller reads the word back when it wants to check.
 *
 * Pages cited (title, then section):
 *   DyLLM        "DyLLM: Efficient Diffusion LLM Inference via Saliency-based
 *                 Token Selection and Partial Attention"
 *   SlowFast     "Accelerating Diffusion Large Language Models with SlowFast
 *                 Sampling: The Three Golden Principles"
 *   Attn-Sampler "Attention-Based Sampler for Diffusion Language Models"
 *   SureLock     "Stopping Computation for Converged Tokens in Masked
 *                 Diffusion-LM Decoding"
 *   LSP          "Beyond Scattered Acceptance: Fast and Coherent Inference for
 *                 DLMs via Longest Stable Prefixes"
 */
#ifndef DLLM_H_
#define DLLM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dllm_status {
  DLLM_OK = 0,
  DLLM_ERR_INVALID_ARG = 1,  /* bad pointer, size, stride or alignment          */
  DLLM_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement     */
  DLLM_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed     */
  DLLM_ERR_DEVICE_CHECK = 4, /* (dev_status only) bad device-side count/index   */
  DLLM_ERR_TIMEOUT = 5       /* (dev_status only) a bounded device wait expired */
} dllm_status;

typedef enum dllm_dtype { DLLM_F32 = 0, DLLM_BF16 = 1 } dllm_dtype;

/* Library version string, e.g. "dllm 0.1.0 sm_103a". */
const char* dllm_version(void);

/* Message of the last failing call on this thread ("" if none). */
const char* dllm_last_error(void);

/*
 * dllm_saliency_select -- temporal cosine saliency, threshold and ordered
 * compaction of the active positions.
 *
 * DyLLM, technical summary, Methodology 1 (layer-adaptive saliency selection):
 * the cosine similarity s of each token's vector at step t and its cached
 * vector at step t-1; a cosine near 1 is stable, a low one is salient and is
 * recomputed.  Methodology 3 (adaptive input): the window scored is the
 * response rows on most steps and the whole sequence every few steps.
 * SureLock, technical summary section 2: locked positions are never active.
 *
 *   cur, prev   [B, Lw, D] of `dtype`; row r of batch b starts at element
 *               b*batch_stride + r*row_stride (row_stride >= D).  Pass the
 *               window's first row as the base pointer.
 *   locked      [B, Lw] uint8 (nonzero = locked), contiguous, or NULL.
 *   tau         threshold: active iff !(cos >= tau) and not locked
 *               (cos == tau is stable; a NaN cosine is salient).
 *   idx_base    added to every emitted index (e.g. the prompt length, so
 *               idx_out holds absolute sequence positions).
 *   cos_out     [B, Lw] float32: cos = <cur,prev> / (|cur| |prev|); both norms
 *               zero -> 1, exactly one zero -> 0.  Float32 accumulation.
 *   idx_out     [B, Lw] int32: ascending active positions + idx_base in
 *               [0, count), then -1.
 *   count_out   [B] int32: number of active positions.
 *
 * Errors: INVALID_ARG for NULL required pointers, B/Lw/D < 1, row_stride < D,
 * batch_stride < Lw*row_stride.  Never touches dev_status (may be NULL).
 */
dllm_status dllm_saliency_select(const void* cur, const void* prev, int dtype,
                                 int B, int Lw, int D, int64_t row_stride,
                                 int64_t batch_stride, const uint8_t* locked,
                                 float tau, int32_t idx_base, float* cos_out,
                                 int32_t* idx_out, int32_t* count_out,
                                 int32_t* dev_status, void* stream);

/*
 * dllm_confidence -- max softmax probability, argmax and logit margin per row.
 *
 * SlowFast, section 2 (certainty principle; the fast phase unmasks tokens
 * whose confidence exceeds a high threshold).  SureLock, technical summary
 * section 2, locking criterion 2: the uncertainty 1 - max_v p(v) (here
 * 1 - conf).  LSP, technical summary section 2 step 1: the logit margin, the
 * highest minus the second-highest logit.
 *
 *   logits      [B, R_src, V] of `dtype`; row r of batch b starts at element
 *               b*batch_stride + r*row_stride (row_stride >= V).
 *   R_max       rows scored per batch row (launch size).
 *   row_idx     [B, R_max] int32 or NULL: row r reads logits row row_idx[b,r]
 *               (must be in [0, R_src)); NULL reads row r, which must lie
 *               below R_src (with count NULL, R_max <= R_src is required; with
 *               count given, R_src may be below R_max -- e.g. a buffer that
 *               holds only the rows a step can have -- and a count above
 *               R_src is a device-side error).
 *   count       [B] int32 or NULL: rows r < count[b] are scored (NULL: all
 *               R_max).  Must lie in [0, R_max].
 *   out_idx     [B, R_max] int32 or NULL: the results of row r land in column
 *               out_idx[b,r] (in [0, out_cols)) of the outputs; NULL: column r
 *               (R_max <= out_cols).
 *   conf_out    [B, out_cols] float32 (batch stride out_cols): max_j softmax_j.
 *   argmax_out  [B, out_cols] int32: lowest index of the maximum logit.
 *   margin_out  [B, out_cols] float32 or NULL: top-1 minus top-2 logit (0 on a
 *               tie for the maximum).
 *   ws          device workspace of at least dllm_confidence_workspace_bytes()
 *               bytes (256-byte aligned); its contents need no initialisation.
 * Columns not written are left untouched.  Logits must be finite.
 * Errors: INVALID_ARG (NULLs, V < 2, R_max < 1, strides, small workspace);
 * dev_status gets DEVICE_CHECK for counts/indices out of range, including a
 * row r >= R_src read without row_idx (row skipped).
 */
size_t dllm_confidence_workspace_bytes(int B, int R_max, int V, int dtype);

dllm_status dllm_confidence(const void* logits, int dtype, int B, int R_src,
                            int V, int64_t row_stride, int64_t batch_stride,
                            int R_max, const int32_t* row_idx,
                            const int32_t* count, const int32_t* out_idx,
                            int out_cols, float* conf_out, int32_t* argmax_out,
                            float* margin_out, void* ws, size_t ws_bytes,
                            int32_t* dev_status, void* stream);

/*
 * dllm_confidence_static_ws -- dllm_confidence for callers that cannot
 * allocate device memory.
 *
 * The pages have no counterpart to this entry point: it exists for callers
 * that only receive their input and output buffers (for instance a plugin
 * that a host framework hands raw device pointers, with no allocator of its
 * own) and for latency-critical callers that cannot afford cudaMalloc, which
 * may synchronise the whole device.  Instead of a caller workspace it uses a
 * scratch array of DLLM_CONFIDENCE_STATIC_WS_BYTES bytes that the library
 * defines in device memory; every GPU that loads the library holds that array
 * until the process exits.
 *
 * Arguments, outputs and device-side checks are those of dllm_confidence,
 * minus ws/ws_bytes.  Rejects (DLLM_ERR_INVALID_ARG, nothing launched) any
 * shape whose scratch need, dllm_confidence_workspace_bytes(B, R_max, V,
 * dtype), exceeds DLLM_CONFIDENCE_STATIC_WS_BYTES.  Allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * The first call on a device (made with that device current) loads the
 * library's module there if CUDA's lazy loading has not yet done so, which
 * creates the array, and looks up the array's device address once; make
 * that first call before any stream capture.  The address is kept for the
 * rest of the process: it belongs to the device's primary context, so after
 * a cudaDeviceReset, or with another context current, it is stale and this
 * entry point must not be used.  All calls on a device share the one array and it keeps the last
 * call's contents: calls whose kernels overlap on the GPU (e.g. on two
 * streams without ordering between them) race on it and must be serialised
 * by the caller.  Nothing in it needs to start at zero: each call writes
 * every partial result it later reads.
 */
#define DLLM_CONFIDENCE_STATIC_WS_BYTES ((size_t)4 << 20) /* 4 MiB */

dllm_status dllm_confidence_static_ws(const void* logits, int dtype, int B,
                                      int R_src, int V, int64_t row_stride,
                                      int64_t batch_stride, int R_max,
                                      const int32_t* row_idx,
                                      const int32_t* count,
                                      const int32_t* out_idx, int out_cols,
                                      float* conf_out, int32_t* argmax_out,
                                      float* margin_out, int32_t* dev_status,
                                      void* stream);

/*
 * dllm_kv_scatter -- write the fresh K/V rows of the active positions into
 * the full-sequence cache.
 *
 * SureLock, technical summary section 2: the K/V of locked positions stay in
 * the cache and active tokens keep attending to them; only active positions
 * get new K/V.  LSP, technical summary section 2 ("KV Cache"): contiguous
 * appends instead of fragmented updates (a run of consecutive indices is the
 * same call).
 *
 *   k_cache, v_cache  [B, L, H, d] of `dtype`, contiguous (updated in place).
 *   k_new, v_new      [B, M_max, H, d], contiguous: row i of batch b is the
 *                     fresh row of position idx[b, i].
 *   idx               [B, M_max] int32: for i < count[b], strictly increasing
 *                     positions in [0, L).
 *   count             [B] int32 in [0, M_max].
 * Every other cache row is left bitwise unchanged.  A row whose index is out
 * of range or not above its predecessor is skipped and dev_status gets
 * DEVICE_CHECK.
 */
dllm_status dllm_kv_scatter(void* k_cache, void* v_cache, const void* k_new,
                            const void* v_new, int dtype, int B, int L, int H,
                            int d, int M_max, const int32_t* idx,
                            const int32_t* count, int32_t* dev_status,
                            void* stream);

/*
 * dllm_partial_attention -- bidirectional attention of the active query rows
 * over the whole cached K/V, with optional per-key column sums.
 *
 * DyLLM, technical summary, Methodology 2 (salient path: score rows of the
 * salient queries are recomputed in full).  SureLock, technical summary
 * section 2: active tokens attend to every position through the cached K/V;
 * cost O(M N d) for M active rows.  Attn-Sampler, technical summary,
 * Methodology 2: column sums of the attention matrix, computed block-wise
 * without materialising it.
 *
 *   q           [B, M_max, H, d] of `dtype`: rows i < count[b] are the active
 *               queries (already projected); rows beyond are ignored.
 *   k_cache, v_cache [B, L, H, d] of `dtype`.
 *   count       [B] int32 in [0, M_max].
 *   scale       score scale; <= 0 selects 1/sqrt(d).
 *   o_out       [B, M_max, H, d] of `dtype`: o_i = sum_j softmax_j(s_i) v_j,
 *               s_ij = scale <q_i, k_j>, no mask; written for rows < count.
 *   lse_out     [B, H, M_max] float32 or NULL: log sum_j exp s_ij (rows <
 *               count).  Required when colsum_out is given.
 *   colsum_out  [B, H, L] float32 or NULL: colsum[b,h,j] = sum over active
 *               rows i of exp(s_ij - lse_i) (written for every j; zero when
 *               count[b] == 0).
 *   ws          workspace of dllm_attention_workspace_bytes() bytes (may be 0).
 * Supported: d in {32, 64, 128} (bf16 d == 128 runs on the tensor cores).
 * Errors: INVALID_ARG, UNSUPPORTED (other d); dev_status gets DEVICE_CHECK for
 * a count outside [0, M_max] (clamped) and TIMEOUT if a bounded pipeline wait
 * expires (that tile's outputs are then not written).
 */
size_t dllm_attention_workspace_bytes(int B, int L, int H, int d, int M_max,
                                      int dtype);

dllm_status dllm_partial_attention(const void* q, const void* k_cache,
                                   const void* v_cache, int dtype, int B, int L,
                                   int H, int d, int M_max,
                                   const int32_t* count, float scale,
                                   void* o_out, float* lse_out,
                                   float* colsum_out, void* ws, size_t ws_bytes,
                                   int32_t* dev_status, void* stream);

/*
 * dllm_attention_colsum -- the per-key column sums alone, from a log-sum-exp
 * computed earlier (the second normalised pass as a call of its own).
 *
 * Attn-Sampler, technical summary, Methodology 2: the column sums of the
 * attention matrix over the active query rows, computed block by block
 * without materialising the matrix.  colsum[b,h,j] = sum over i < count[b] of
 * exp(scale <q_i, k_j> - lse[b,h,i]); with the lse that
 * dllm_partial_attention wrote for the same q, k_cache and scale, this is
 * exactly the colsum_out that call computes.
 *
 *   q, k_cache, count, scale, B, L, H, d, M_max  as in dllm_partial_attention.
 *   lse         [B, H, M_max] float32 (rows < count[b] are read).
 *   colsum_out  [B, H, L] float32, written for every j (zero when
 *               count[b] == 0).
 * Errors as dllm_partial_attention.
 */
dllm_status dllm_attention_colsum(const void* q, const void* k_cache, int dtype,
                                  int B, int L, int H, int d, int M_max,
                                  const int32_t* count, float scale,
                                  const float* lse, float* colsum_out,
                                  int32_t* dev_status, void* stream);

/*
 * dllm_stable_prefix -- length of the longest stable block at the head of
 * the remaining active suffix.
 *
 * LSP, technical summary section 2: commit the longest contiguous stable
 * block at the start of the remaining active sequence in one step, judged by
 * a per-position stability score (step 1); step 4 (fallback) commits at least
 * one token when none is stable.
 *
 *   score       [B, L] float32, contiguous: position p is stable iff
 *               score[b,p] >= tau (NaN is unstable).  Callers write +inf at
 *               positions that must count as stable (already committed).
 *   start       [B] int32 in [0, L]: first position of the remaining suffix.
 *   min_commit  nonzero: a zero length becomes 1 when start < L.
 *   advance_start nonzero: start[b] += len[b] after the scan (start is then
 *               written).
 *   len_out     [B] int32.
 * Errors: INVALID_ARG; dev_status gets DEVICE_CHECK for start outside [0, L]
 * (len 0, start unchanged).
 */
dllm_status dllm_stable_prefix(const float* score, int B, int L, int32_t* start,
                               float tau, int min_commit, int advance_start,
                               int32_t* len_out, int32_t* dev_status,
                               void* stream);

/*
 * dllm_lock_criterion -- SureLock's locking criterion: the local KL
 * divergence of each row's predictive distribution between the previous and
 * the current step, its uncertainty, and the lock flags.
 *
 * SureLock, technical summary section 2, locking criterion 1: a position
 * locks when D = KL(p_t || p_{t-1}) falls below eps; criterion 2 (optional
 * gate): its uncertainty 1 - max_v p_t(v) must lie below a percentile.  The
 * percentile is taken over the active rows of the same batch row: with n
 * active rows and gate fraction q in (0, 1) the gate passes iff the
 * uncertainty is at most the k-th smallest one, k = max(1, ceil(q n)) (q as
 * float32, the product exact); q <= 0 or q >= 1 disables the gate.
 *
 *   logits_cur, logits_prev  [B, R_src, V] of `dtype`, the same layout
 *               (row r of batch b at b*batch_stride + r*row_stride): the
 *               current and the previous step's logits of the same rows.
 *   R_max, row_idx, count, out_idx, out_cols  as in dllm_confidence.
 *   eps         KL threshold: a row locks iff kl < eps (float32 compare) and
 *               the gate passes; NaN never locks.
 *   kl_out      [B, out_cols] float32: sum_j p_j (log p_j - log q_j),
 *               p = softmax(current row), q = softmax(previous row).
 *   unc_out     [B, out_cols] float32: 1 - max_j p_j.
 *   locked_inout [B, out_cols] uint8 or NULL: set to 1 at the columns of the
 *               rows that lock (never cleared: a lock is permanent); usable
 *               as the `locked` mask of dllm_saliency_select.  R_max must be
 *               at most 16384 when it is given.
 *   ws          workspace of dllm_lock_workspace_bytes() bytes (16-byte
 *               aligned); its contents need no initialisation.
 * Logits must be finite.  Errors: INVALID_ARG (NULLs, sizes, strides, small
 * workspace, R_max above 16384 with lock flags); dev_status gets
 * DEVICE_CHECK for counts/indices out of range (row skipped).
 */
size_t dllm_lock_workspace_bytes(int B, int R_max, int V, int dtype);

dllm_status dllm_lock_criterion(const void* logits_cur, const void* logits_prev,
                                int dtype, int B, int R_src, int V,
                                int64_t row_stride, int64_t batch_stride,
                                int R_max, const int32_t* row_idx,
                                const int32_t* count, const int32_t* out_idx,
                                int out_cols, float eps, float gate_q,
                                float* kl_out, float* unc_out,
                                uint8_t* locked_inout, void* ws,
                                size_t ws_bytes, int32_t* dev_status,
                                void* stream);

/*
 * dllm_lock_criterion_conf -- dllm_lock_criterion and the confidence of the
 * current rows (dllm_confidence's outputs) from one read of the logits.
 *
 * SureLock, technical summary section 2: criterion 2's uncertainty is
 * 1 - max_v p_t(v), the complement of the confidence that SlowFast (section
 * 2, certainty principle) and LSP (technical summary section 2, step 1, with
 * the logit margin) score the same rows by; both criteria read the current
 * step's logits, so one pass over them yields every output.
 *
 *   Arguments as in dllm_lock_criterion (same workspace size), plus
 *   conf_out    [B, out_cols] float32: max_j softmax_j of the current row.
 *   argmax_out  [B, out_cols] int32: lowest index of its maximum logit.
 *   margin_out  [B, out_cols] float32 or NULL: top-1 minus top-2 logit (0 on
 *               a tie for the maximum).
 * The columns written are those of kl_out, and conf_out equals 1 - unc_out
 * before the clamp at 0.  V must be at least 2.  Errors: as
 * dllm_lock_criterion, and INVALID_ARG for NULL conf_out or argmax_out.
 */
dllm_status dllm_lock_criterion_conf(const void* logits_cur,
                                     const void* logits_prev, int dtype, int B,
                                     int R_src, int V, int64_t row_stride,
                                     int64_t batch_stride, int R_max,
                                     const int32_t* row_idx,
                                     const int32_t* count,
                                     const int32_t* out_idx, int out_cols,
                                     float eps, float gate_q, float* kl_out,
                                     float* unc_out, float* conf_out,
                                     int32_t* argmax_out, float* margin_out,
                                     uint8_t* locked_inout, void* ws,
                                     size_t ws_bytes, int32_t* dev_status,
                                     void* stream);

/*
 * dllm_adaptive_prefix -- the longest stable prefix with an adaptive
 * threshold.
 *
 * LSP, technical summary section 2, step 2 (adaptive sizing): instead of a
 * fixed threshold, tau is chosen so that the committed stable block covers a
 * fraction [lo, hi] of the current active length A = L - start; step 4
 * (fallback): at least one token.  With the prefix minima
 * m_k = min(score[start .. start + k - 1]) (NaN counts as -inf),
 * k_lo = max(1, ceil(lo A)), k_hi = max(k_lo, floor(hi A)) (float32 lo, hi;
 * exact products): tau = m_{k_lo}; len = min(k_hi, #{k : m_k >= tau}),
 * never past the first NaN score, at least 1 when A > 0.
 *
 *   score       [B, L] float32, contiguous (e.g. the logit margin of
 *               dllm_confidence, +inf at committed positions).
 *   start       [B] int32 in [0, L]; advance_start nonzero: start += len.
 *   lo, hi      fractions in [0, 1].
 *   len_out     [B] int32 (0 when A = 0).
 *   tau_out     [B] float32: the threshold chosen (+inf when A = 0).
 * Errors: INVALID_ARG; dev_status gets DEVICE_CHECK for start outside
 * [0, L] (len 0).
 */
dllm_status dllm_adaptive_prefix(const float* score, int B, int L,
                                 int32_t* start, float lo, float hi,
                                 int advance_start, int32_t* len_out,
                                 float* tau_out, int32_t* dev_status,
                                 void* stream);

/*
 * dllm_attn_scores -- total attention each position receives.
 *
 * Attn-Sampler, technical summary, Methodology 1 (decode in descending order
 * of the column sums of the attention matrix) and the ablation on layers and
 * heads (aggregate over all of them):
 *   score[b, j] (+)= sum_h colsum[b, h, j], heads added in order 0 .. H-1.
 *
 *   colsum      [B, H, L] float32, contiguous (the column sums of
 *               dllm_partial_attention or dllm_attention_colsum).
 *   accumulate  nonzero: add onto score_inout (the sum over layers is one
 *               call per layer); zero: overwrite it.
 *   score_inout [B, L] float32, contiguous.
 * Errors: INVALID_ARG (NULLs, sizes, B above 65535).  dev_status is unused
 * (no device-side index is read) and may be NULL.
 */
dllm_status dllm_attn_scores(const float* colsum, int B, int H, int L,
                             int accumulate, float* score_inout,
                             int32_t* dev_status, void* stream);

/*
 * dllm_attn_sampler_select -- decoding order and the number of tokens to
 * decode in parallel.
 *
 * Attn-Sampler, technical summary, Methodology 2: the tokens with the highest
 * scores are decoded first, and in parallel only while their score exceeds a
 * threshold.  The page does not give the dynamic threshold; here it is
 * thr = max(tau, gamma * score of the top candidate) for gamma > 0 (product
 * rounded to float32; a NaN top leaves tau), else tau.
 *
 *   score       [B, L] float32, contiguous (e.g. from dllm_attn_scores).
 *   candidates  [B, L] uint8, nonzero where a position may be decoded (still
 *               masked), or NULL for all positions.
 *   k_max       cap on the count when > 0.
 *   order_out   [B, L] int32: the candidates by descending score, equal scores
 *               by ascending position (-0 equals +0, NaN last), then -1.
 *   n_out       [B] int32: the number of leading entries of order_out whose
 *               score is >= thr, capped at k_max, at least 1 when there is a
 *               candidate, 0 when there is none.
 * L at most 16384.  Errors: INVALID_ARG (NULLs, sizes, NaN tau or gamma).
 * dev_status is unused and may be NULL.
 */
dllm_status dllm_attn_sampler_select(const float* score, int B, int L,
                                     const uint8_t* candidates, float tau,
                                     float gamma, int k_max,
                                     int32_t* order_out, int32_t* n_out,
                                     int32_t* dev_status, void* stream);

/*
 * dllm_approx_attention_update -- output update of the stable rows from the
 * value changes of the salient rows.
 *
 * DyLLM, technical summary, Methodology 2 (non-salient path): a stable row
 * keeps its attention weights, and its output moves by the change of the
 * salient tokens' values weighted by them; cost O(N |A|).  The weights are
 * the previous step's, recovered from the cached query, the previous keys of
 * the salient positions and the cached log-sum-exp:
 *   o[i] += sum_{a < count} exp(scale q[i].k[idx_a] - lse[i]) (v_new[a] - v[idx_a])
 * for every stable position i = stable_idx[r], r < stable_count.
 *
 *   q_prev, k_prev, v_prev  [B, L, H, d] of `dtype`, contiguous: the previous
 *               step's queries, keys and values of every position (k_prev
 *               and v_prev before this step's dllm_kv_scatter).
 *   lse_prev    [B, H, L] float32: the previous step's log-sum-exp of every
 *               position's score row.
 *   v_new       [B, M_max, H, d]: row a is the fresh value of position
 *               idx[b, a], a < count[b] (the layout of dllm_kv_scatter).
 *   idx, count  [B, M_max], [B] int32: the salient positions.
 *   stable_idx, stable_count  [B, N_max], [B] int32: distinct positions
 *               whose outputs are updated.
 *   scale       <= 0 selects 1/sqrt(d).
 *   o_inout     [B, L, H, d] of `dtype`: outputs by position, updated in
 *               place on the stable rows only (float32 arithmetic, rounded to
 *               the dtype once).
 * d in {32, 64, 128}.  Errors: INVALID_ARG, UNSUPPORTED (head dim);
 * dev_status gets DEVICE_CHECK for counts or positions out of range (the
 * row or column is skipped).
 */
dllm_status dllm_approx_attention_update(const void* q_prev,
                                         const float* lse_prev,
                                         const void* k_prev, const void* v_prev,
                                         const void* v_new, int dtype, int B,
                                         int L, int H, int d, int M_max,
                                         const int32_t* idx,
                                         const int32_t* count, int N_max,
                                         const int32_t* stable_idx,
                                         const int32_t* stable_count,
                                         float scale, void* o_inout,
                                         int32_t* dev_status, void* stream);

/*
 * dllm_snap_prefix -- structural snapping of the committed block.
 *
 * LSP, technical summary section 2, step 3: the end of the selected block
 * moves to the nearest natural boundary (punctuation, newline, code symbol)
 * inside the candidate block.  The block [start[b], start[b] + len[b]) ends
 * after its last boundary token at a position >= start + max(min_len, 1) - 1:
 * len becomes that position - start + 1; with no such token len is kept.
 *
 *   tokens      [B, L] int32, contiguous: the token at each position (e.g.
 *               argmax_out of dllm_confidence).
 *   delim       [V] uint8: nonzero for the vocabulary ids that are
 *               boundaries (the tokenizer's punctuation, newline, code
 *               symbols; supplied by the caller).
 *   start       [B] int32; len_inout [B] int32 (e.g. from
 *               dllm_adaptive_prefix), updated in place.
 *   min_len     the shortest block snapping may leave (e.g. the lower end of
 *               the adaptive range).
 * Errors: INVALID_ARG; dev_status gets DEVICE_CHECK for a block outside
 * [0, L] (left as it is) or a token outside [0, V) (not a boundary).
 */
dllm_status dllm_snap_prefix(const int32_t* tokens, int B, int L, int V,
                             const uint8_t* delim, const int32_t* start,
                             int32_t* len_inout, int min_len,
                             int32_t* dev_status, void* stream);

/*
 * SlowFast phase control (host side).
 *
 * SlowFast, section 2 (pipeline): the slow phase watches the prediction of
 * the convergence point e_cand over a sliding window of steps; once its
 * variance falls below sigma^2_stable the region [s_cycle, e_cycle] is
 * stable and the fast phase decodes it (every masked token of the region
 * above the high confidence threshold at once); then a new cycle begins.
 *
 * The controller keeps, per batch row, the predictions of the current cycle
 * (at most `window`).  dllm_slowfast_observe appends this step's prediction;
 * the step is fast iff the window is full, the latest prediction lies beyond
 * start[b], and W sum x^2 - (sum x)^2 < sigma2 W^2 (the population variance
 * below sigma2, left side exact in 64-bit integers, right side in double).
 * A fast step reports phase 1 and region [start[b], e_cand[b]) and empties
 * the window; otherwise phase 0 and region end -1.
 *
 * All pointers of these three calls are HOST memory: start, e_cand,
 * phase_out, region_end_out are [B] int32 arrays.  e_cand is typically
 * start + the stable-prefix length of the confidence scores from start
 * (dllm_stable_prefix with the confidence threshold), read back by the
 * caller.  A handle is not thread-safe; create returns INVALID_ARG for
 * B < 1, window < 1 or sigma2 < 0 (or NaN).
 */
typedef struct dllm_slowfast dllm_slowfast;

/*
 * dllm_slowfast_observe_device -- the same controller with its state and its
 * per-step arrays in device memory, as a kernel on `stream`, so that a
 * decoding loop reads nothing back to the host (SlowFast, section 2,
 * pipeline, as above).
 *
 *   state       int32 device array of dllm_slowfast_state_bytes(B, window)
 *               bytes, zeroed by the caller before the first step of a
 *               sequence: per batch row the number of predictions held,
 *               then those predictions, oldest first.  Owned by the caller;
 *               reuse it only with the same B and window.
 *   start       [B] int32 (device): the start of the undecoded suffix.
 *   pred_len    [B] int32 (device): the convergence prediction of this step
 *               as a length from start, e_cand = start + pred_len (e.g.
 *               len_out of dllm_stable_prefix over the confidence scores
 *               with the convergence threshold, advance_start = 0).
 *   phase_out, region_end_out  [B] int32 (device): as dllm_slowfast_observe.
 * window <= 4096.  Errors: INVALID_ARG (NULLs, B or window < 1, window above
 * 4096, sigma2 < 0 or NaN); dev_status gets DEVICE_CHECK for a state word
 * out of range (that row's cycle restarts).
 */
size_t dllm_slowfast_state_bytes(int B, int window);

dllm_status dllm_slowfast_observe_device(int32_t* state, int B, int window,
                                         double sigma2_stable,
                                         const int32_t* start,
                                         const int32_t* pred_len,
                                         int32_t* phase_out,
                                         int32_t* region_end_out,
                                         int32_t* dev_status, void* stream);

/*
 * dllm_slowfast_select -- the tokens a SlowFast step unmasks.
 *
 * SlowFast, section 2 (pipeline): the exploratory (slow) phase selects the
 * tokens with the highest confidence in an exploration window; the
 * accelerated (fast) phase unmasks at once every masked token of the stable
 * region [s_cycle, e_cycle] whose confidence exceeds tau_high_conf.  Per
 * batch row b, on the device:
 *   phase[b] == 1 (fast): the still-masked positions p in
 *     [start[b], region_end[b]) with conf[b,p] > tau_high (float32, NaN
 *     never passes); no fallback (none may pass).
 *   otherwise (slow): the min(k, candidates) still-masked positions of the
 *     window [start[b], start[b] + width) cut at L with the highest
 *     confidence, equal confidences by lower position, NaN never selected.
 *
 *   conf        [B, L] float32, contiguous (e.g. conf_out of dllm_confidence).
 *   masked      [B, L] uint8 (nonzero = still masked) or NULL (all masked).
 *   start, phase, region_end  [B] int32 (device): phase and region as
 *               dllm_slowfast_observe(_device) reports them.
 *   tau_high    fast-phase threshold; width in [1, 16384]; k in [1, 64].
 *   idx_out     [B, L] int32: the selected positions in ascending order,
 *               then -1.
 *   count_out   [B] int32: how many.
 * Errors: INVALID_ARG (NULLs, sizes, NaN tau_high); dev_status gets
 * DEVICE_CHECK for start outside [0, L] (nothing selected) or a fast
 * region_end outside [start, L] (clamped).
 */
dllm_status dllm_slowfast_select(const float* conf, const uint8_t* masked,
                                 int B, int L, const int32_t* start,
                                 const int32_t* phase, const int32_t* region_end,
                                 float tau_high, int width, int k,
                                 int32_t* idx_out, int32_t* count_out,
                                 int32_t* dev_status, void* stream);

dllm_status dllm_slowfast_create(int B, int window, double sigma2_stable,
                                 dllm_slowfast** out);

dllm_status dllm_slowfast_observe(dllm_slowfast* sf, const int32_t* start,
                                  const int32_t* e_cand, int32_t* phase_out,
                                  int32_t* region_end_out);

void dllm_slowfast_destroy(dllm_slowfast* sf);

/*
 * Diagnostics.  None computes anything of the step; they let tests check
 * the library's own machinery and give the bench its reference for the
 * memory-bound calls.  The pages have no counterpart to them.
 *
 * dllm_exp2_fma_eval -- y[i] = 2^x[i] through the FMA-pipe exponential the
 * attention kernels use for part of their exponentials (Cody-Waite split
 * x = n + f, n = round(x), and a degree-4 minimax polynomial for 2^f; x is
 * clamped at -125 and must be at most 128).  x, y: n float32 in device
 * memory.  Errors: INVALID_ARG (NULLs, n < 1), CUDA (launch).
 *
 * dllm_set_wait_limit -- the clock cycles after which a bounded pipeline wait
 * of the streaming confidence kernel and of the attention forward kernel
 * gives up for kernels launched after this call (process-wide; 0 restores
 * the default of about a second).  A wait that runs out records
 * DLLM_ERR_TIMEOUT in dev_status; the kernel then waits (with the default
 * limit) for its own copies and tensor-core work in flight, frees its tensor
 * memory and returns, leaving that call's outputs incomplete.  For tests of
 * that path; not thread-safe against concurrent launches.  Errors:
 * INVALID_ARG for a negative count.
 *
 * dllm_read_stream -- reads `bytes` bytes of `buf` (device memory, 16-byte
 * aligned, bytes a positive multiple of 16) once, in one launch of one
 * persistent CTA per SM that copies 32 KB chunks into a four-stage
 * shared-memory ring with cp.async.bulk and computes nothing: its duration is
 * the time one launch of a read-bound kernel of that size needs at least on
 * this GPU, launch, ramp-up and tail included, the reference the memory-bound
 * calls are measured against.  A byte of each chunk is added into *sink (one
 * uint32 in device memory, accumulated with atomicAdd) so that the copies are
 * observable.  A pipeline wait that runs out records DLLM_ERR_TIMEOUT in
 * *dev_status.  Errors: INVALID_ARG (NULLs, size, alignment), CUDA (launch).
 */
dllm_status dllm_exp2_fma_eval(const float* x, float* y, int n, void* stream);

dllm_status dllm_set_wait_limit(long long cycles);

dllm_status dllm_read_stream(const void* buf, size_t bytes, uint32_t* sink,
                             int32_t* dev_status, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* DLLM_H_ */
