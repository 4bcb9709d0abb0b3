// Launchers behind the C ABI.  Each returns the cudaError_t of its launches;
// arguments were validated by the entry points in api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dllm {

cudaError_t launch_saliency_select(const void* cur, const void* prev, int dtype, int B,
                                   int Lw, int D, int64_t row_stride, int64_t batch_stride,
                                   const uint8_t* locked, float tau, int32_t idx_base,
                                   float* cos_out, int32_t* idx_out, int32_t* count_out,
                                   cudaStream_t stream);

size_t confidence_workspace_bytes(int B, int R_max, int V, int dtype);

cudaError_t launch_confidence(const void* logits, int dtype, int B, int R_src, int V,
                              int64_t row_stride, int64_t batch_stride, int R_max,
                              const int32_t* row_idx, const int32_t* count,
                              const int32_t* out_idx, int out_cols, float* conf_out,
                              int32_t* argmax_out, float* margin_out, void* ws,
                              int32_t* dev_status, cudaStream_t stream);

cudaError_t launch_kv_scatter(void* k_cache, void* v_cache, const void* k_new,
                              const void* v_new, int dtype, int B, int L, int H, int d,
                              int M_max, const int32_t* idx, const int32_t* count,
                              int32_t* dev_status, cudaStream_t stream);

size_t attention_workspace_bytes(int B, int L, int H, int d, int M_max, int dtype);

cudaError_t launch_attention_simt(const void* q, const void* k, const void* v, int dtype,
                                  int B, int L, int H, int d, int M_max, const int32_t* count,
                                  float scale, void* o, float* lse, int32_t* dev_status,
                                  cudaStream_t stream);

bool attention_tc_supported(int dtype, int d, const void* q, const void* k, const void* v,
                            const void* o);

size_t attention_tc_workspace_bytes(int n_ctas);

cudaError_t launch_attention_tc(const void* q, const void* k, const void* v, int B, int L, int H,
                                int M_max, const int32_t* count, float scale, void* o, float* lse,
                                float* colsum, void* ws, size_t ws_bytes, int32_t* dev_status,
                                cudaStream_t stream);

cudaError_t launch_colsum_tc(const void* q, const void* k, int B, int L, int H, int M_max,
                             const int32_t* count, float scale, const float* lse, float* colsum,
                             int32_t* dev_status, cudaStream_t stream);

cudaError_t launch_colsum_simt(const void* q, const void* k, int dtype, int B, int L, int H,
                               int d, int M_max, const int32_t* count, float scale,
                               const float* lse, float* colsum, int32_t* dev_status,
                               cudaStream_t stream);

cudaError_t launch_stable_prefix(const float* score, int B, int L, int32_t* start, float tau,
                                 int min_commit, int advance_start, int32_t* len_out,
                                 int32_t* dev_status, cudaStream_t stream);

size_t lock_workspace_bytes(int B, int R_max, int V, int dtype);

cudaError_t launch_lock_criterion(const void* z, const void* y, int dtype, int B, int R_src,
                                  int V, int64_t rs, int64_t bs, int R_max,
                                  const int32_t* row_idx, const int32_t* count,
                                  const int32_t* out_idx, int out_cols, float eps, float gate_q,
                                  float* kl_out, float* unc_out, float* conf_out,
                                  int32_t* argmax_out, float* margin_out, uint8_t* locked,
                                  void* ws, int32_t* dev_status, cudaStream_t stream);

cudaError_t launch_adaptive_prefix(const float* score, int B, int L, int32_t* start, float lo,
                                   float hi, int advance_start, int32_t* len_out, float* tau_out,
                                   int32_t* dev_status, cudaStream_t stream);

cudaError_t launch_attn_scores(const float* colsum, int B, int H, int L, int accumulate,
                               float* score, cudaStream_t stream);

int attn_sampler_max_len();

cudaError_t launch_attn_sampler_select(const float* score, int B, int L,
                                       const uint8_t* candidates, float tau, float gamma,
                                       int k_max, int32_t* order, int32_t* n_out,
                                       cudaStream_t stream);

cudaError_t launch_approx_attention_update(const void* q, const float* lse, const void* k,
                                           const void* v, const void* v_new, int dtype, int B,
                                           int L, int H, int d, int M_max, const int32_t* idx,
                                           const int32_t* count, int N_max,
                                           const int32_t* stable_idx,
                                           const int32_t* stable_count, float scale, void* o,
                                           int32_t* dev_status, cudaStream_t stream);

bool approx_update_tc_supported(int dtype, int d, const void* q, const void* k, const void* v,
                                const void* v_new, const void* o);

cudaError_t launch_approx_update_tc(const void* q, const float* lse, const void* k, const void* v,
                                    const void* v_new, int B, int L, int H, int M_max,
                                    const int32_t* idx, const int32_t* count, int N_max,
                                    const int32_t* stable_idx, const int32_t* stable_count,
                                    float scale, void* o, int32_t* dev_status,
                                    cudaStream_t stream);

cudaError_t launch_snap_prefix(const int32_t* tokens, int B, int L, int V, const uint8_t* delim,
                               const int32_t* start, int32_t* len, int min_len,
                               int32_t* dev_status, cudaStream_t stream);

int slowfast_select_max_width();

cudaError_t launch_slowfast_observe(int32_t* state, int B, int W, double sigma2,
                                    const int32_t* start, const int32_t* pred_len,
                                    int32_t* phase_out, int32_t* region_end_out,
                                    int32_t* dev_status, cudaStream_t stream);

cudaError_t launch_slowfast_select(const float* conf, const uint8_t* masked, int B, int L,
                                   const int32_t* start, const int32_t* phase,
                                   const int32_t* region_end, float tau_high, int width, int k,
                                   int32_t* idx_out, int32_t* count_out, int32_t* dev_status,
                                   cudaStream_t stream);

int num_sms();

// Clock cycles a bounded pipeline wait of the streaming confidence and the
// attention forward kernels may take before it gives up (dllm_set_wait_limit).
long long wait_limit();

// Raises the dynamic shared-memory limit of `func` to `bytes` on the current
// device (once per function and device: later calls keep the first value, so
// a kernel whose size varies passes its largest size).
cudaError_t ensure_smem_limit(const void* func, int bytes);

// Records `message` as the thread's dllm_last_error() text and returns `code`.
int set_last_error(int code, const char* message);

}  // namespace dllm
