// Temporal cosine saliency and ordered compaction of the active positions.
//
// DyLLM ("Efficient Diffusion LLM Inference via Saliency-based Token Selection
// and Partial Attention"), technical summary, Methodology 1: per token, the
// cosine similarity of its vector at step t and the cached vector of step t-1;
// high similarity is stable, low similarity is salient and gets recomputed.
// SureLock, technical summary section 2: locked positions are never active.
//
// Two launches:
//   cos_rows_kernel  one warp per row, 16-byte streaming loads, three float32
//                    accumulators (<a,b>, |a|^2, |b|^2) reduced by shuffles.
//                    HBM bound: 2 * D * sizeof(T) bytes per row.
//   compact_kernel   one CTA per batch row: threshold + lock mask, block-wide
//                    exclusive scan, ascending idx, -1 padding, count.
#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kCosWarps = 8;   // warps (rows in flight) per CTA
constexpr int kCosUnroll = 4;  // 16-byte vectors per operand per lane in flight

template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int kElems = 4;
  static __device__ __forceinline__ void acc(const uint4& a, const uint4& b, float& dot,
                                             float& na, float& nb) {
    const float x[4] = {__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z),
                        __uint_as_float(a.w)};
    const float y[4] = {__uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z),
                        __uint_as_float(b.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      dot = fmaf(x[i], y[i], dot);
      na = fmaf(x[i], x[i], na);
      nb = fmaf(y[i], y[i], nb);
    }
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int kElems = 8;
  static __device__ __forceinline__ void acc(const uint4& a, const uint4& b, float& dot,
                                             float& na, float& nb) {
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
    const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float x0 = bf16_lo(wa[i]), x1 = bf16_hi(wa[i]);
      const float y0 = bf16_lo(wb[i]), y1 = bf16_hi(wb[i]);
      dot = fmaf(x0, y0, dot);
      dot = fmaf(x1, y1, dot);
      na = fmaf(x0, x0, na);
      na = fmaf(x1, x1, na);
      nb = fmaf(y0, y0, nb);
      nb = fmaf(y1, y1, nb);
    }
  }
};

__device__ __forceinline__ float cosine_from_sums(float dot, float na, float nb) {
  if (na == 0.0f && nb == 0.0f) return 1.0f;  // two zero vectors are identical
  if (na == 0.0f || nb == 0.0f) return 0.0f;  // a zero vector is orthogonal to all
  return dot / (sqrtf(na) * sqrtf(nb));
}

// VEC: rows are 16-byte aligned and D is a multiple of the vector width.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kCosWarps * 32)
cos_rows_kernel(const T* __restrict__ cur, const T* __restrict__ prev, int B, int Lw, int D,
                int64_t rs, int64_t bs, float* __restrict__ cos_out) {
  const int lane = threadIdx.x & 31;
  const int64_t total = (int64_t)B * Lw;
  const int64_t stride = (int64_t)gridDim.x * kCosWarps;
  for (int64_t row = (int64_t)blockIdx.x * kCosWarps + (threadIdx.x >> 5); row < total;
       row += stride) {
    const int b = (int)(row / Lw);
    const int r = (int)(row - (int64_t)b * Lw);
    const T* pc = cur + b * bs + r * rs;
    const T* pp = prev + b * bs + r * rs;
    float dot = 0.f, na = 0.f, nb = 0.f;
    if constexpr (VEC) {
      constexpr int E = Vec16<T>::kElems;
      const int nvec = D / E;
      const uint4* vc = reinterpret_cast<const uint4*>(pc);
      const uint4* vp = reinterpret_cast<const uint4*>(pp);
      for (int base = 0; base < nvec; base += 32 * kCosUnroll) {
        uint4 a[kCosUnroll], c[kCosUnroll];
#pragma unroll
        for (int u = 0; u < kCosUnroll; ++u) {
          const int v = base + u * 32 + lane;
          if (v < nvec) {
            a[u] = ld_stream16(vc + v);
            c[u] = ld_stream16(vp + v);
          } else {
            a[u] = make_uint4(0, 0, 0, 0);
            c[u] = make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int u = 0; u < kCosUnroll; ++u) Vec16<T>::acc(a[u], c[u], dot, na, nb);
      }
    } else {
      for (int k = lane; k < D; k += 32) {
        const float x = Elem<T>::to_f32(pc[k]);
        const float y = Elem<T>::to_f32(pp[k]);
        dot = fmaf(x, y, dot);
        na = fmaf(x, x, na);
        nb = fmaf(y, y, nb);
      }
    }
    dot = warp_sum(dot);
    na = warp_sum(na);
    nb = warp_sum(nb);
    if (lane == 0) cos_out[row] = cosine_from_sums(dot, na, nb);
  }
}

constexpr int kCompactThreads = 1024;
constexpr int kCompactItems = 4;  // consecutive positions per thread per chunk

__global__ void __launch_bounds__(kCompactThreads)
compact_kernel(const float* __restrict__ cos, const uint8_t* __restrict__ locked, int Lw,
               float tau, int32_t idx_base, int32_t* __restrict__ idx_out,
               int32_t* __restrict__ count_out) {
  __shared__ int warp_tot[kCompactThreads / 32];
  __shared__ int chunk_total;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* c = cos + (int64_t)b * Lw;
  const uint8_t* lk = locked ? locked + (int64_t)b * Lw : nullptr;
  int32_t* out = idx_out + (int64_t)b * Lw;
  int running = 0;
  for (int start = 0; start < Lw; start += kCompactThreads * kCompactItems) {
    bool act[kCompactItems];
    int mine = 0;
#pragma unroll
    for (int k = 0; k < kCompactItems; ++k) {
      const int p = start + tid * kCompactItems + k;
      bool a = false;
      if (p < Lw) {
        a = !(c[p] >= tau);  // NaN cosine counts as salient
        if (lk != nullptr && lk[p] != 0) a = false;
      }
      act[k] = a;
      mine += a ? 1 : 0;
    }
    // inclusive warp scan of per-thread counts
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = lane < kCompactThreads / 32 ? warp_tot[lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      if (lane < kCompactThreads / 32) warp_tot[lane] = wi - w;  // exclusive
      if (lane == 31) chunk_total = wi;
    }
    __syncthreads();
    int pos = running + warp_tot[warp] + incl - mine;
#pragma unroll
    for (int k = 0; k < kCompactItems; ++k) {
      if (act[k]) out[pos++] = start + tid * kCompactItems + k + idx_base;
    }
    running += chunk_total;
    __syncthreads();  // warp_tot / chunk_total are rewritten by the next chunk
  }
  for (int p = running + tid; p < Lw; p += kCompactThreads) out[p] = -1;
  if (tid == 0) count_out[b] = running;
}

template <typename T>
cudaError_t launch_typed(const T* cur, const T* prev, int B, int Lw, int D, int64_t rs,
                         int64_t bs, float* cos_out, cudaStream_t stream) {
  const int64_t rows = (int64_t)B * Lw;
  const int64_t want = (rows + kCosWarps - 1) / kCosWarps;
  const int grid = (int)(want < (int64_t)num_sms() * 16 ? want : (int64_t)num_sms() * 16);
  constexpr int E = 16 / sizeof(T);
  const bool vec = (reinterpret_cast<uintptr_t>(cur) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(prev) % 16 == 0) && (D % E == 0) &&
                   (rs % E == 0) && (bs % E == 0);
  if (vec)
    cos_rows_kernel<T, true><<<grid, kCosWarps * 32, 0, stream>>>(cur, prev, B, Lw, D, rs, bs,
                                                                  cos_out);
  else
    cos_rows_kernel<T, false><<<grid, kCosWarps * 32, 0, stream>>>(cur, prev, B, Lw, D, rs, bs,
                                                                   cos_out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_saliency_select(const void* cur, const void* prev, int dtype, int B,
                                   int Lw, int D, int64_t row_stride, int64_t batch_stride,
                                   const uint8_t* locked, float tau, int32_t idx_base,
                                   float* cos_out, int32_t* idx_out, int32_t* count_out,
                                   cudaStream_t stream) {
  cudaError_t e;
  if (dtype == DLLM_BF16)
    e = launch_typed(static_cast<const __nv_bfloat16*>(cur),
                     static_cast<const __nv_bfloat16*>(prev), B, Lw, D, row_stride,
                     batch_stride, cos_out, stream);
  else
    e = launch_typed(static_cast<const float*>(cur), static_cast<const float*>(prev), B, Lw, D,
                     row_stride, batch_stride, cos_out, stream);
  if (e != cudaSuccess) return e;
  compact_kernel<<<B, kCompactThreads, 0, stream>>>(cos_out, locked, Lw, tau, idx_base, idx_out,
                                                    count_out);
  return cudaGetLastError();
}

}  // namespace dllm
