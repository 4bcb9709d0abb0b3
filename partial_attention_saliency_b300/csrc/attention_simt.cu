// Partial attention and column sums on the CUDA cores (float32 arithmetic).
//
// Serves float32 tensors and head dims the tensor-core kernel does not take
// (d = 32, 64, and float32 d = 128).
//
// DyLLM ("Efficient Diffusion LLM Inference via Saliency-based Token Selection
// and Partial Attention"), technical summary, Methodology 2: the score rows of
// the salient (active) queries are recomputed in full.  SureLock, technical
// summary section 2: active rows attend to every position via the cached K/V.
// Attn-Sampler, technical summary, Methodology 2: per-key column sums of the
// attention matrix, computed block by block.
//
// attn_simt_kernel: one CTA per (16 active query rows, head, batch); key tiles
// of 32 rows staged in shared memory as float32; each warp keeps 4 query rows
// with an online (running max / running sum) softmax; lane j scores key j of
// the tile, and the P V product broadcasts p_j with shuffles.
//
// colsum_simt_kernel: one CTA per (32 keys, head, batch); lane j owns key j,
// the four warps split the active query rows; p_ij = exp(s_ij - lse_i) is
// summed in a fixed order (no atomics, run-to-run identical).
#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kQT = 16;  // query rows per CTA
constexpr int kKT = 32;  // keys per tile
constexpr int kWarps = 4;
constexpr int kRowsPerWarp = kQT / kWarps;

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
attn_simt_kernel(const T* q, const T* k, const T* v,
                 int L, int H, int M_max, const int32_t* count, float scale_log2,
                 T* o, float* lse, int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  __shared__ float Qs[kQT][D];
  __shared__ float Ks[kKT][D + 1];
  __shared__ float Vs[kKT][D];
  const int h = blockIdx.y, b = blockIdx.z;
  const int i0 = blockIdx.x * kQT;
  int n = __ldca(count + b);
  if (n < 0 || n > M_max) {
    if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
    n = n < 0 ? 0 : M_max;
  }
  if (i0 >= n) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t hd = (int64_t)H * D;

  for (int e = tid; e < kQT * D; e += kWarps * 32) {
    const int r = e / D, t = e - r * D;
    const int i = i0 + r;
    Qs[r][t] = i < n ? Elem<T>::to_f32(__ldca(q + ((int64_t)b * M_max + i) * hd + (int64_t)h * D + t)) : 0.f;
  }

  constexpr int C = D / 32;  // output dims per lane
  float acc[kRowsPerWarp][C];
  float m[kRowsPerWarp], l[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) acc[r][c] = 0.f;
  }

  for (int j0 = 0; j0 < L; j0 += kKT) {
    __syncthreads();  // previous tile fully consumed (and Qs visible on the first pass)
    for (int e = tid; e < kKT * D; e += kWarps * 32) {
      const int j = e / D, t = e - j * D;
      const int jj = j0 + j;
      float kv = 0.f, vv = 0.f;
      if (jj < L) {
        const int64_t off = ((int64_t)b * L + jj) * hd + (int64_t)h * D + t;
        kv = Elem<T>::to_f32(__ldca(k + off));
        vv = Elem<T>::to_f32(__ldca(v + off));
      }
      Ks[j][t] = kv;
      Vs[j][t] = vv;
    }
    __syncthreads();
    const bool key_ok = (j0 + lane) < L;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int qr = warp * kRowsPerWarp + r;
      float dot = 0.f;
#pragma unroll 8
      for (int t = 0; t < D; ++t) dot = fmaf(Qs[qr][t], Ks[lane][t], dot);
      const float s = key_ok ? dot * scale_log2 : -INFINITY;
      const float m_new = fmaxf(m[r], warp_max(s));
      const float alpha = ex2_approx(m[r] - m_new);
      const float p = ex2_approx(s - m_new);
      l[r] = l[r] * alpha + warp_sum(p);
      m[r] = m_new;
#pragma unroll
      for (int c = 0; c < C; ++c) acc[r][c] *= alpha;
      for (int j = 0; j < kKT; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int c = 0; c < C; ++c) acc[r][c] = fmaf(pj, Vs[j][lane + 32 * c], acc[r][c]);
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = i0 + warp * kRowsPerWarp + r;
    if (i >= n) continue;
    const float inv = 1.0f / l[r];
    T* orow = o + ((int64_t)b * M_max + i) * hd + (int64_t)h * D;
#pragma unroll
    for (int c = 0; c < C; ++c) orow[lane + 32 * c] = Elem<T>::from_f32(acc[r][c] * inv);
    if (lse != nullptr && lane == 0)
      lse[((int64_t)b * H + h) * M_max + i] = (m[r] + log2f(l[r])) * 0.69314718055994531f;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
colsum_simt_kernel(const T* q, const T* k, int L, int H, int M_max,
                   const int32_t* count, float scale_log2,
                   const float* lse, float* colsum) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  __shared__ float Ks[kKT][D + 1];
  __shared__ float Qs[kQT][D];
  __shared__ float Ls[kQT];
  __shared__ float part[kWarps][kKT];
  const int h = blockIdx.y, b = blockIdx.z;
  const int j0 = blockIdx.x * kKT;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int n = __ldca(count + b);
  n = n < 0 ? 0 : (n > M_max ? M_max : n);
  const int64_t hd = (int64_t)H * D;
  for (int e = tid; e < kKT * D; e += kWarps * 32) {
    const int j = e / D, t = e - j * D;
    const int jj = j0 + j;
    Ks[j][t] = jj < L ? Elem<T>::to_f32(__ldca(k + ((int64_t)b * L + jj) * hd + (int64_t)h * D + t)) : 0.f;
  }
  float acc = 0.f;
  for (int i0 = 0; i0 < n; i0 += kQT) {
    __syncthreads();
    for (int e = tid; e < kQT * D; e += kWarps * 32) {
      const int r = e / D, t = e - r * D;
      const int i = i0 + r;
      Qs[r][t] = i < n ? Elem<T>::to_f32(__ldca(q + ((int64_t)b * M_max + i) * hd + (int64_t)h * D + t)) : 0.f;
    }
    if (tid < kQT) {
      const int i = i0 + tid;
      Ls[tid] = i < n ? __ldca(lse + ((int64_t)b * H + h) * M_max + i) * kLog2e : INFINITY;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int qr = warp * kRowsPerWarp + r;
      float dot = 0.f;
#pragma unroll 8
      for (int t = 0; t < D; ++t) dot = fmaf(Qs[qr][t], Ks[lane][t], dot);
      acc += ex2_approx(dot * scale_log2 - Ls[qr]);  // rows past n carry lse = +inf -> 0
    }
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    const float s = ((part[0][lane] + part[1][lane]) + part[2][lane]) + part[3][lane];
    const int j = j0 + lane;
    if (j < L) colsum[((int64_t)b * H + h) * L + j] = s;
  }
}

template <typename T, int D>
cudaError_t launch_attn(const void* q, const void* k, const void* v, int B, int L, int H,
                        int M_max, const int32_t* count, float scale, void* o, float* lse,
                        int32_t* dev_status, cudaStream_t stream) {
  dim3 grid((M_max + kQT - 1) / kQT, H, B);
  launch_pdl(attn_simt_kernel<T, D>, grid, kWarps * 32, 0, stream,
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), L, H, M_max,
      count, scale * kLog2e, static_cast<T*>(o), lse, dev_status);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_cs(const void* q, const void* k, int B, int L, int H, int M_max,
                      const int32_t* count, float scale, const float* lse, float* colsum,
                      cudaStream_t stream) {
  dim3 grid((L + kKT - 1) / kKT, H, B);
  launch_pdl(colsum_simt_kernel<T, D>, grid, kWarps * 32, 0, stream,
      static_cast<const T*>(q), static_cast<const T*>(k), L, H, M_max, count, scale * kLog2e, lse,
      colsum);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_simt(const void* q, const void* k, const void* v, int dtype,
                                  int B, int L, int H, int d, int M_max, const int32_t* count,
                                  float scale, void* o, float* lse, int32_t* dev_status,
                                  cudaStream_t stream) {
  if (dtype == DLLM_BF16) {
    if (d == 32) return launch_attn<__nv_bfloat16, 32>(q, k, v, B, L, H, M_max, count, scale, o, lse, dev_status, stream);
    if (d == 64) return launch_attn<__nv_bfloat16, 64>(q, k, v, B, L, H, M_max, count, scale, o, lse, dev_status, stream);
    return launch_attn<__nv_bfloat16, 128>(q, k, v, B, L, H, M_max, count, scale, o, lse, dev_status, stream);
  }
  if (d == 32) return launch_attn<float, 32>(q, k, v, B, L, H, M_max, count, scale, o, lse, dev_status, stream);
  if (d == 64) return launch_attn<float, 64>(q, k, v, B, L, H, M_max, count, scale, o, lse, dev_status, stream);
  return launch_attn<float, 128>(q, k, v, B, L, H, M_max, count, scale, o, lse, dev_status, stream);
}

cudaError_t launch_colsum_simt(const void* q, const void* k, int dtype, int B, int L, int H,
                               int d, int M_max, const int32_t* count, float scale,
                               const float* lse, float* colsum, int32_t* /*dev_status*/,
                               cudaStream_t stream) {
  if (dtype == DLLM_BF16) {
    if (d == 32) return launch_cs<__nv_bfloat16, 32>(q, k, B, L, H, M_max, count, scale, lse, colsum, stream);
    if (d == 64) return launch_cs<__nv_bfloat16, 64>(q, k, B, L, H, M_max, count, scale, lse, colsum, stream);
    return launch_cs<__nv_bfloat16, 128>(q, k, B, L, H, M_max, count, scale, lse, colsum, stream);
  }
  if (d == 32) return launch_cs<float, 32>(q, k, B, L, H, M_max, count, scale, lse, colsum, stream);
  if (d == 64) return launch_cs<float, 64>(q, k, B, L, H, M_max, count, scale, lse, colsum, stream);
  return launch_cs<float, 128>(q, k, B, L, H, M_max, count, scale, lse, colsum, stream);
}

}  // namespace dllm
