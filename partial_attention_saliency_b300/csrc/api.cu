// extern "C" entry points of libdllm: argument validation, launch, error text.
//
// Nothing here allocates device memory, synchronises a stream or reads device
// data: counts stay on the device and the kernels read them there.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <set>
#include <string>
#include <utility>

#include "dllm.h"
#include "internal.h"

namespace dllm {

int num_sms() {
  static thread_local int cached_dev = -1;
  static thread_local int cached_sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cached_sms;
  if (dev != cached_dev) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
      cached_sms = sms;
    cached_dev = dev;
  }
  return cached_sms;
}

cudaError_t ensure_smem_limit(const void* func, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({func, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({func, dev});
  return e;
}

}  // namespace dllm

namespace {

thread_local std::string g_last_error;

dllm_status fail(dllm_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

dllm_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return DLLM_OK;
  return fail(DLLM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool valid_dtype(int dt) { return dt == DLLM_F32 || dt == DLLM_BF16; }

#define REQUIRE(cond, ...)                                   \
  do {                                                       \
    if (!(cond)) return fail(DLLM_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

// The checks and the launch of dllm_lock_criterion and dllm_lock_criterion_conf
// (conf_out NULL: the criterion alone).
dllm_status lock_criterion_call(const char* name, const void* logits_cur,
                                const void* logits_prev, int dtype, int B, int R_src, int V,
                                int64_t row_stride, int64_t batch_stride, int R_max,
                                const int32_t* row_idx, const int32_t* count,
                                const int32_t* out_idx, int out_cols, float eps, float gate_q,
                                float* kl_out, float* unc_out, float* conf_out,
                                int32_t* argmax_out, float* margin_out, uint8_t* locked_inout,
                                void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  REQUIRE(logits_cur && logits_prev && kl_out && unc_out, "%s: NULL logits or output pointer",
          name);
  REQUIRE(valid_dtype(dtype), "%s: unknown dtype %d", name, dtype);
  REQUIRE(B >= 1 && R_src >= 1 && R_max >= 1, "%s: B=%d R_src=%d R_max=%d", name, B, R_src,
          R_max);
  REQUIRE(V >= 1, "%s: V=%d must be >= 1", name, V);
  REQUIRE(row_stride >= V, "%s: row_stride %lld < V", name, (long long)row_stride);
  REQUIRE(B == 1 || batch_stride >= (int64_t)R_src * row_stride, "%s: batch_stride too small",
          name);
  // as in dllm_confidence: rows past R_src without row_idx are caught on the device
  REQUIRE(row_idx != nullptr || count != nullptr || R_max <= R_src,
          "%s: R_max > R_src without row_idx or count", name);
  REQUIRE(out_cols >= 1 && (out_idx != nullptr || R_max <= out_cols), "%s: out_cols %d too small",
          name, out_cols);
  REQUIRE(locked_inout == nullptr || R_max <= 16384, "%s: R_max %d above 16384 with lock flags",
          name, R_max);
  REQUIRE((int64_t)B * R_max <= 2147483647, "%s: B*R_max too large", name);
  const size_t need = dllm::lock_workspace_bytes(B, R_max, V, dtype);
  REQUIRE(ws != nullptr && ws_bytes >= need, "%s: workspace %zu bytes < %zu required", name,
          ws_bytes, need);
  REQUIRE(reinterpret_cast<uintptr_t>(ws) % 16 == 0, "%s: workspace misaligned", name);
  return from_cuda(dllm::launch_lock_criterion(logits_cur, logits_prev, dtype, B, R_src, V,
                                               row_stride, batch_stride, R_max, row_idx, count,
                                               out_idx, out_cols, eps, gate_q, kl_out, unc_out,
                                               conf_out, argmax_out, margin_out, locked_inout,
                                               ws, dev_status, static_cast<cudaStream_t>(stream)),
                   "lock criterion launch");
}

}  // namespace

extern "C" {

const char* dllm_version(void) { return "dllm 0.1.0 sm_103a"; }

const char* dllm_last_error(void) { return g_last_error.c_str(); }

dllm_status dllm_saliency_select(const void* cur, const void* prev, int dtype, int B, int Lw,
                                 int D, int64_t row_stride, int64_t batch_stride,
                                 const uint8_t* locked, float tau, int32_t idx_base,
                                 float* cos_out, int32_t* idx_out, int32_t* count_out,
                                 int32_t* dev_status, void* stream) {
  (void)dev_status;
  REQUIRE(cur && prev && cos_out && idx_out && count_out,
          "dllm_saliency_select: NULL input or output pointer");
  REQUIRE(valid_dtype(dtype), "dllm_saliency_select: unknown dtype %d", dtype);
  REQUIRE(B >= 1 && Lw >= 1 && D >= 1, "dllm_saliency_select: B=%d Lw=%d D=%d must be >= 1", B,
          Lw, D);
  REQUIRE(row_stride >= D, "dllm_saliency_select: row_stride %lld < D %d",
          (long long)row_stride, D);
  REQUIRE(B == 1 || batch_stride >= (int64_t)Lw * row_stride,
          "dllm_saliency_select: batch_stride %lld < Lw*row_stride", (long long)batch_stride);
  REQUIRE((int64_t)idx_base + Lw <= INT32_MAX && idx_base >= 0,
          "dllm_saliency_select: idx_base %d out of range", idx_base);
  return from_cuda(dllm::launch_saliency_select(cur, prev, dtype, B, Lw, D, row_stride,
                                                batch_stride, locked, tau, idx_base, cos_out,
                                                idx_out, count_out,
                                                static_cast<cudaStream_t>(stream)),
                   "dllm_saliency_select launch");
}

size_t dllm_confidence_workspace_bytes(int B, int R_max, int V, int dtype) {
  if (B < 1 || R_max < 1 || V < 1 || !valid_dtype(dtype)) return 0;
  return dllm::confidence_workspace_bytes(B, R_max, V, dtype);
}

dllm_status dllm_confidence(const void* logits, int dtype, int B, int R_src, int V,
                            int64_t row_stride, int64_t batch_stride, int R_max,
                            const int32_t* row_idx, const int32_t* count,
                            const int32_t* out_idx, int out_cols, float* conf_out,
                            int32_t* argmax_out, float* margin_out, void* ws, size_t ws_bytes,
                            int32_t* dev_status, void* stream) {
  REQUIRE(logits && conf_out && argmax_out, "dllm_confidence: NULL logits or output pointer");
  REQUIRE(valid_dtype(dtype), "dllm_confidence: unknown dtype %d", dtype);
  REQUIRE(B >= 1 && R_src >= 1 && R_max >= 1, "dllm_confidence: B=%d R_src=%d R_max=%d", B,
          R_src, R_max);
  REQUIRE(V >= 2, "dllm_confidence: V=%d must be >= 2", V);
  REQUIRE(row_stride >= V, "dllm_confidence: row_stride %lld < V", (long long)row_stride);
  REQUIRE(B == 1 || batch_stride >= (int64_t)R_src * row_stride,
          "dllm_confidence: batch_stride too small");
  // Without row_idx, rows r < count[b] are read; a count above R_src is caught on the device
  // (DEVICE_CHECK, the rows past R_src skipped), so only a call that scores all R_max rows
  // needs R_max <= R_src here.
  REQUIRE(row_idx != nullptr || count != nullptr || R_max <= R_src,
          "dllm_confidence: R_max > R_src without row_idx or count");
  REQUIRE(out_cols >= 1 && (out_idx != nullptr || R_max <= out_cols),
          "dllm_confidence: out_cols %d too small", out_cols);
  const size_t need = dllm::confidence_workspace_bytes(B, R_max, V, dtype);
  REQUIRE(ws != nullptr && ws_bytes >= need,
          "dllm_confidence: workspace %zu bytes < %zu required", ws_bytes, need);
  REQUIRE(reinterpret_cast<uintptr_t>(ws) % 16 == 0, "dllm_confidence: workspace misaligned");
  REQUIRE((int64_t)B * R_max <= INT32_MAX, "dllm_confidence: B*R_max too large");
  return from_cuda(dllm::launch_confidence(logits, dtype, B, R_src, V, row_stride, batch_stride,
                                           R_max, row_idx, count, out_idx, out_cols, conf_out,
                                           argmax_out, margin_out, ws, dev_status,
                                           static_cast<cudaStream_t>(stream)),
                   "dllm_confidence launch");
}

dllm_status dllm_kv_scatter(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                            int dtype, int B, int L, int H, int d, int M_max,
                            const int32_t* idx, const int32_t* count, int32_t* dev_status,
                            void* stream) {
  REQUIRE(k_cache && v_cache && k_new && v_new && idx && count,
          "dllm_kv_scatter: NULL pointer argument");
  REQUIRE(valid_dtype(dtype), "dllm_kv_scatter: unknown dtype %d", dtype);
  REQUIRE(B >= 1 && L >= 1 && H >= 1 && d >= 1 && M_max >= 1,
          "dllm_kv_scatter: B=%d L=%d H=%d d=%d M_max=%d must be >= 1", B, L, H, d, M_max);
  REQUIRE(B <= 65535, "dllm_kv_scatter: B=%d exceeds 65535", B);
  return from_cuda(dllm::launch_kv_scatter(k_cache, v_cache, k_new, v_new, dtype, B, L, H, d,
                                           M_max, idx, count, dev_status,
                                           static_cast<cudaStream_t>(stream)),
                   "dllm_kv_scatter launch");
}

size_t dllm_attention_workspace_bytes(int B, int L, int H, int d, int M_max, int dtype) {
  if (B < 1 || L < 1 || H < 1 || d < 1 || M_max < 1 || !valid_dtype(dtype)) return 0;
  return dllm::attention_workspace_bytes(B, L, H, d, M_max, dtype);
}

dllm_status dllm_partial_attention(const void* q, const void* k_cache, const void* v_cache,
                                   int dtype, int B, int L, int H, int d, int M_max,
                                   const int32_t* count, float scale, void* o_out,
                                   float* lse_out, float* colsum_out, void* ws,
                                   size_t ws_bytes, int32_t* dev_status, void* stream) {
  REQUIRE(q && k_cache && v_cache && count && o_out,
          "dllm_partial_attention: NULL pointer argument");
  REQUIRE(valid_dtype(dtype), "dllm_partial_attention: unknown dtype %d", dtype);
  REQUIRE(B >= 1 && L >= 1 && H >= 1 && M_max >= 1,
          "dllm_partial_attention: B=%d L=%d H=%d M_max=%d must be >= 1", B, L, H, M_max);
  REQUIRE(B <= 65535 && H <= 65535, "dllm_partial_attention: B or H above 65535");
  REQUIRE(colsum_out == nullptr || lse_out != nullptr,
          "dllm_partial_attention: colsum_out needs lse_out");
  if (d != 32 && d != 64 && d != 128)
    return fail(DLLM_ERR_UNSUPPORTED, "dllm_partial_attention: head dim %d not in {32,64,128}", d);
  if (ws_bytes > 0 && ws == nullptr)
    return fail(DLLM_ERR_INVALID_ARG, "dllm_partial_attention: ws_bytes > 0 with a NULL workspace");
  if (!(scale > 0.0f)) scale = 1.0f / std::sqrt((float)d);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dllm::attention_tc_supported(dtype, d, q, k_cache, v_cache, o_out)) {
    return from_cuda(dllm::launch_attention_tc(q, k_cache, v_cache, B, L, H, M_max, count, scale,
                                               o_out, lse_out, colsum_out, ws, ws_bytes,
                                               dev_status, s),
                     "dllm_partial_attention launch");
  }
  cudaError_t e = dllm::launch_attention_simt(q, k_cache, v_cache, dtype, B, L, H, d, M_max,
                                              count, scale, o_out, lse_out, dev_status, s);
  if (e != cudaSuccess) return from_cuda(e, "dllm_partial_attention launch");
  if (colsum_out != nullptr) {
    e = dllm::launch_colsum_simt(q, k_cache, dtype, B, L, H, d, M_max, count, scale, lse_out,
                                 colsum_out, dev_status, s);
    if (e != cudaSuccess) return from_cuda(e, "dllm_partial_attention column-sum launch");
  }
  return DLLM_OK;
}

dllm_status dllm_attention_colsum(const void* q, const void* k_cache, int dtype, int B, int L,
                                  int H, int d, int M_max, const int32_t* count, float scale,
                                  const float* lse, float* colsum_out, int32_t* dev_status,
                                  void* stream) {
  REQUIRE(q && k_cache && count && lse && colsum_out,
          "dllm_attention_colsum: NULL pointer argument");
  REQUIRE(valid_dtype(dtype), "dllm_attention_colsum: unknown dtype %d", dtype);
  REQUIRE(B >= 1 && L >= 1 && H >= 1 && M_max >= 1,
          "dllm_attention_colsum: B=%d L=%d H=%d M_max=%d must be >= 1", B, L, H, M_max);
  REQUIRE(B <= 65535 && H <= 65535, "dllm_attention_colsum: B or H above 65535");
  if (d != 32 && d != 64 && d != 128)
    return fail(DLLM_ERR_UNSUPPORTED, "dllm_attention_colsum: head dim %d not in {32,64,128}", d);
  if (!(scale > 0.0f)) scale = 1.0f / std::sqrt((float)d);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dllm::attention_tc_supported(dtype, d, q, k_cache, k_cache, q))
    return from_cuda(dllm::launch_colsum_tc(q, k_cache, B, L, H, M_max, count, scale, lse,
                                            colsum_out, dev_status, s),
                     "dllm_attention_colsum launch");
  return from_cuda(dllm::launch_colsum_simt(q, k_cache, dtype, B, L, H, d, M_max, count, scale,
                                            lse, colsum_out, dev_status, s),
                   "dllm_attention_colsum launch");
}

dllm_status dllm_stable_prefix(const float* score, int B, int L, int32_t* start, float tau,
                               int min_commit, int advance_start, int32_t* len_out,
                               int32_t* dev_status, void* stream) {
  REQUIRE(score && start && len_out, "dllm_stable_prefix: NULL pointer argument");
  REQUIRE(B >= 1 && L >= 1, "dllm_stable_prefix: B=%d L=%d must be >= 1", B, L);
  return from_cuda(dllm::launch_stable_prefix(score, B, L, start, tau, min_commit, advance_start,
                                              len_out, dev_status,
                                              static_cast<cudaStream_t>(stream)),
                   "dllm_stable_prefix launch");
}

size_t dllm_lock_workspace_bytes(int B, int R_max, int V, int dtype) {
  if (B < 1 || R_max < 1 || V < 1 || !valid_dtype(dtype)) return 0;
  return dllm::lock_workspace_bytes(B, R_max, V, dtype);
}

dllm_status dllm_lock_criterion(const void* logits_cur, const void* logits_prev, int dtype,
                                int B, int R_src, int V, int64_t row_stride,
                                int64_t batch_stride, int R_max, const int32_t* row_idx,
                                const int32_t* count, const int32_t* out_idx, int out_cols,
                                float eps, float gate_q, float* kl_out, float* unc_out,
                                uint8_t* locked_inout, void* ws, size_t ws_bytes,
                                int32_t* dev_status, void* stream) {
  return lock_criterion_call("dllm_lock_criterion", logits_cur, logits_prev, dtype, B, R_src, V,
                             row_stride, batch_stride, R_max, row_idx, count, out_idx, out_cols,
                             eps, gate_q, kl_out, unc_out, nullptr, nullptr, nullptr,
                             locked_inout, ws, ws_bytes, dev_status, stream);
}

dllm_status dllm_lock_criterion_conf(const void* logits_cur, const void* logits_prev, int dtype,
                                     int B, int R_src, int V, int64_t row_stride,
                                     int64_t batch_stride, int R_max, const int32_t* row_idx,
                                     const int32_t* count, const int32_t* out_idx, int out_cols,
                                     float eps, float gate_q, float* kl_out, float* unc_out,
                                     float* conf_out, int32_t* argmax_out, float* margin_out,
                                     uint8_t* locked_inout, void* ws, size_t ws_bytes,
                                     int32_t* dev_status, void* stream) {
  REQUIRE(conf_out && argmax_out, "dllm_lock_criterion_conf: NULL conf_out or argmax_out");
  REQUIRE(V >= 2, "dllm_lock_criterion_conf: V=%d must be >= 2", V);
  return lock_criterion_call("dllm_lock_criterion_conf", logits_cur, logits_prev, dtype, B, R_src,
                             V, row_stride, batch_stride, R_max, row_idx, count, out_idx,
                             out_cols, eps, gate_q, kl_out, unc_out, conf_out, argmax_out,
                             margin_out, locked_inout, ws, ws_bytes, dev_status, stream);
}

dllm_status dllm_adaptive_prefix(const float* score, int B, int L, int32_t* start, float lo,
                                 float hi, int advance_start, int32_t* len_out, float* tau_out,
                                 int32_t* dev_status, void* stream) {
  REQUIRE(score && start && len_out && tau_out, "dllm_adaptive_prefix: NULL pointer argument");
  REQUIRE(B >= 1 && L >= 1, "dllm_adaptive_prefix: B=%d L=%d must be >= 1", B, L);
  REQUIRE(L < (1 << 29), "dllm_adaptive_prefix: L=%d too large", L);
  REQUIRE(lo >= 0.0f && lo <= 1.0f && hi >= 0.0f && hi <= 1.0f,
          "dllm_adaptive_prefix: fractions lo=%g hi=%g outside [0, 1]", lo, hi);
  return from_cuda(dllm::launch_adaptive_prefix(score, B, L, start, lo, hi, advance_start,
                                                len_out, tau_out, dev_status,
                                                static_cast<cudaStream_t>(stream)),
                   "dllm_adaptive_prefix launch");
}

dllm_status dllm_attn_scores(const float* colsum, int B, int H, int L, int accumulate,
                             float* score_inout, int32_t* dev_status, void* stream) {
  (void)dev_status;  // nothing is read through device-side indices
  REQUIRE(colsum && score_inout, "dllm_attn_scores: NULL pointer argument");
  REQUIRE(B >= 1 && H >= 1 && L >= 1, "dllm_attn_scores: B=%d H=%d L=%d must be >= 1", B, H, L);
  REQUIRE(B <= 65535, "dllm_attn_scores: B=%d above 65535", B);
  return from_cuda(dllm::launch_attn_scores(colsum, B, H, L, accumulate, score_inout,
                                            static_cast<cudaStream_t>(stream)),
                   "dllm_attn_scores launch");
}

dllm_status dllm_attn_sampler_select(const float* score, int B, int L,
                                     const uint8_t* candidates, float tau, float gamma,
                                     int k_max, int32_t* order_out, int32_t* n_out,
                                     int32_t* dev_status, void* stream) {
  (void)dev_status;  // nothing is read through device-side indices
  REQUIRE(score && order_out && n_out, "dllm_attn_sampler_select: NULL pointer argument");
  REQUIRE(B >= 1 && L >= 1, "dllm_attn_sampler_select: B=%d L=%d must be >= 1", B, L);
  REQUIRE(L <= dllm::attn_sampler_max_len(), "dllm_attn_sampler_select: L=%d above %d", L,
          dllm::attn_sampler_max_len());
  REQUIRE(!std::isnan(tau) && !std::isnan(gamma),
          "dllm_attn_sampler_select: NaN threshold or fraction");
  return from_cuda(dllm::launch_attn_sampler_select(score, B, L, candidates, tau, gamma, k_max,
                                                    order_out, n_out,
                                                    static_cast<cudaStream_t>(stream)),
                   "dllm_attn_sampler_select launch");
}

dllm_status dllm_approx_attention_update(const void* q_prev, const float* lse_prev,
                                         const void* k_prev, const void* v_prev,
                                         const void* v_new, int dtype, int B, int L, int H, int d,
                                         int M_max, const int32_t* idx, const int32_t* count,
                                         int N_max, const int32_t* stable_idx,
                                         const int32_t* stable_count, float scale, void* o_inout,
                                         int32_t* dev_status, void* stream) {
  REQUIRE(q_prev && lse_prev && k_prev && v_prev && v_new && idx && count && stable_idx &&
              stable_count && o_inout,
          "dllm_approx_attention_update: NULL pointer argument");
  REQUIRE(valid_dtype(dtype), "dllm_approx_attention_update: unknown dtype %d", dtype);
  REQUIRE(B >= 1 && L >= 1 && H >= 1 && M_max >= 1 && N_max >= 1,
          "dllm_approx_attention_update: B=%d L=%d H=%d M_max=%d N_max=%d must be >= 1", B, L, H,
          M_max, N_max);
  REQUIRE(B <= 65535 && H <= 65535, "dllm_approx_attention_update: B=%d or H=%d above 65535", B,
          H);
  if (d != 32 && d != 64 && d != 128)
    return fail(DLLM_ERR_UNSUPPORTED, "dllm_approx_attention_update: head dim %d not in {32, 64, 128}",
                d);
  if (!(scale > 0.0f)) scale = 1.0f / std::sqrt((float)d);
  return from_cuda(dllm::launch_approx_attention_update(
                       q_prev, lse_prev, k_prev, v_prev, v_new, dtype, B, L, H, d, M_max, idx,
                       count, N_max, stable_idx, stable_count, scale, o_inout, dev_status,
                       static_cast<cudaStream_t>(stream)),
                   "dllm_approx_attention_update launch");
}

dllm_status dllm_snap_prefix(const int32_t* tokens, int B, int L, int V, const uint8_t* delim,
                             const int32_t* start, int32_t* len_inout, int min_len,
                             int32_t* dev_status, void* stream) {
  REQUIRE(tokens && delim && start && len_inout, "dllm_snap_prefix: NULL pointer argument");
  REQUIRE(B >= 1 && L >= 1 && V >= 1, "dllm_snap_prefix: B=%d L=%d V=%d must be >= 1", B, L, V);
  return from_cuda(dllm::launch_snap_prefix(tokens, B, L, V, delim, start, len_inout, min_len,
                                            dev_status, static_cast<cudaStream_t>(stream)),
                   "dllm_snap_prefix launch");
}

size_t dllm_slowfast_state_bytes(int B, int window) {
  if (B < 1 || window < 1) return 0;
  return (size_t)B * (size_t)(window + 1) * sizeof(int32_t);
}

dllm_status dllm_slowfast_observe_device(int32_t* state, int B, int window, double sigma2_stable,
                                         const int32_t* start, const int32_t* pred_len,
                                         int32_t* phase_out, int32_t* region_end_out,
                                         int32_t* dev_status, void* stream) {
  REQUIRE(state && start && pred_len && phase_out && region_end_out,
          "dllm_slowfast_observe_device: NULL pointer argument");
  REQUIRE(B >= 1 && window >= 1, "dllm_slowfast_observe_device: B=%d window=%d must be >= 1", B,
          window);
  REQUIRE(window <= 4096, "dllm_slowfast_observe_device: window %d above 4096", window);
  REQUIRE(sigma2_stable >= 0.0, "dllm_slowfast_observe_device: sigma2 must be >= 0");
  return from_cuda(dllm::launch_slowfast_observe(state, B, window, sigma2_stable, start, pred_len,
                                                 phase_out, region_end_out, dev_status,
                                                 static_cast<cudaStream_t>(stream)),
                   "dllm_slowfast_observe_device launch");
}

dllm_status dllm_slowfast_select(const float* conf, const uint8_t* masked, int B, int L,
                                 const int32_t* start, const int32_t* phase,
                                 const int32_t* region_end, float tau_high, int width, int k,
                                 int32_t* idx_out, int32_t* count_out, int32_t* dev_status,
                                 void* stream) {
  REQUIRE(conf && start && phase && region_end && idx_out && count_out,
          "dllm_slowfast_select: NULL pointer argument");
  REQUIRE(B >= 1 && B <= 65535 && L >= 1, "dllm_slowfast_select: B=%d L=%d out of range", B, L);
  REQUIRE(width >= 1 && width <= dllm::slowfast_select_max_width(),
          "dllm_slowfast_select: width %d outside [1, %d]", width,
          dllm::slowfast_select_max_width());
  REQUIRE(k >= 1 && k <= 64, "dllm_slowfast_select: k %d outside [1, 64]", k);
  REQUIRE(!std::isnan(tau_high), "dllm_slowfast_select: NaN tau_high");
  return from_cuda(dllm::launch_slowfast_select(conf, masked, B, L, start, phase, region_end,
                                                tau_high, width, k, idx_out, count_out,
                                                dev_status, static_cast<cudaStream_t>(stream)),
                   "dllm_slowfast_select launch");
}

}  // extern "C"

namespace dllm {
size_t attention_workspace_bytes(int, int, int, int d, int, int dtype) {
  // only the tensor-core path uses a workspace (key-range split partials)
  return (dtype == DLLM_BF16 && d == 128) ? attention_tc_workspace_bytes(num_sms()) : 0;
}

int set_last_error(int code, const char* message) {
  g_last_error = message;
  return code;
}
}  // namespace dllm
