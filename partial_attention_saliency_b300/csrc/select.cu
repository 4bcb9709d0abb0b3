// Temporal cosine saliency and ordered compaction of the active positions.
//
// DyLLM ("Efficient Diffusion LLM Inference via Saliency-based Token Selection
// and Partial Attention"), technical summary, Methodology 1: per token, the
// cosine similarity of its vector at step t and the cached vector of step t-1;
// high similarity is stable, low similarity is salient and gets recomputed.
// SureLock, technical summary section 2: locked positions are never active.
//
// Two launches:
//   cos_rows_kernel  32 to 256 threads per row (more when rows are few),
//                    16-byte streaming loads, three float32 accumulators
//                    (<a,b>, |a|^2, |b|^2) reduced by shuffles.
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

// One group of TPR threads (TPR in {32, 64, 128, 256}) per row, 256 threads
// per CTA.  Few rows (a 512-row window) take 256 threads each so that every
// SM streams; many rows take one warp each.  VEC: rows are 16-byte aligned and
// D is a multiple of the vector width.
template <typename T, bool VEC, int TPR>
__global__ void __launch_bounds__(kCosWarps * 32)
cos_rows_kernel(const T* cur, const T* prev, int B, int Lw, int D,
                int64_t rs, int64_t bs, float* cos_out) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  constexpr int kRowsPerCta = kCosWarps * 32 / TPR;
  constexpr int kWarpsPerRow = TPR / 32;
  __shared__ float red[kCosWarps][3];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gi = threadIdx.x / TPR;  // row slot in the CTA
  const int li = threadIdx.x % TPR;  // thread within the row group
  const int64_t total = (int64_t)B * Lw;
  for (int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta; row0 < total;
       row0 += (int64_t)gridDim.x * kRowsPerCta) {
    const int64_t row = row0 + gi;
    float dot = 0.f, na = 0.f, nb = 0.f;
    if (row < total) {
      const int b = (int)(row / Lw);
      const int r = (int)(row - (int64_t)b * Lw);
      const T* pc = cur + b * bs + r * rs;
      const T* pp = prev + b * bs + r * rs;
      if constexpr (VEC) {
        constexpr int E = Vec16<T>::kElems;
        const int nvec = D / E;
        const uint4* vc = reinterpret_cast<const uint4*>(pc);
        const uint4* vp = reinterpret_cast<const uint4*>(pp);
        for (int base = 0; base < nvec; base += TPR * kCosUnroll) {
          uint4 a[kCosUnroll], c[kCosUnroll];
#pragma unroll
          for (int u = 0; u < kCosUnroll; ++u) {
            const int v = base + u * TPR + li;
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
        for (int k = li; k < D; k += TPR) {
          const float x = Elem<T>::to_f32(pc[k]);
          const float y = Elem<T>::to_f32(pp[k]);
          dot = fmaf(x, y, dot);
          na = fmaf(x, x, na);
          nb = fmaf(y, y, nb);
        }
      }
    }
    dot = warp_sum(dot);
    na = warp_sum(na);
    nb = warp_sum(nb);
    if constexpr (kWarpsPerRow == 1) {
      if (lane == 0 && row < total) cos_out[row] = cosine_from_sums(dot, na, nb);
    } else {
      if (lane == 0) {
        red[warp][0] = dot;
        red[warp][1] = na;
        red[warp][2] = nb;
      }
      __syncthreads();
      if (li == 0 && row < total) {
        float sd = 0.f, sa = 0.f, sb = 0.f;
#pragma unroll
        for (int w = 0; w < kWarpsPerRow; ++w) {  // fixed order: run-to-run identical
          sd += red[gi * kWarpsPerRow + w][0];
          sa += red[gi * kWarpsPerRow + w][1];
          sb += red[gi * kWarpsPerRow + w][2];
        }
        cos_out[row] = cosine_from_sums(sd, sa, sb);
      }
      __syncthreads();
    }
  }
}

constexpr int kCompactThreads = 1024;
constexpr int kCompactItems = 4;  // consecutive positions per thread per chunk

__global__ void __launch_bounds__(kCompactThreads)
compact_kernel(const float* cos, const uint8_t* locked, int Lw,
               float tau, int32_t idx_base, int32_t* idx_out,
               int32_t* count_out) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
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
        a = !(__ldca(c + p) >= tau);  // NaN cosine counts as salient
        if (lk != nullptr && __ldca(lk + p) != 0) a = false;
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

template <typename T, bool VEC, int TPR>
void launch_cos(const T* cur, const T* prev, int B, int Lw, int D, int64_t rs, int64_t bs,
                float* cos_out, cudaStream_t stream) {
  constexpr int kRowsPerCta = kCosWarps * 32 / TPR;
  const int64_t rows = (int64_t)B * Lw;
  const int64_t want = (rows + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t cap = (int64_t)num_sms() * 16;
  const int grid = (int)(want < cap ? want : cap);
  launch_pdl(cos_rows_kernel<T, VEC, TPR>, grid, kCosWarps * 32, 0, stream, cur, prev, B, Lw, D, rs, bs,
                                                                    cos_out);
}

template <typename T, bool VEC>
void launch_cos_tpr(const T* cur, const T* prev, int B, int Lw, int D, int64_t rs, int64_t bs,
                    float* cos_out, cudaStream_t stream) {
  // enough row groups for ~16 resident warps per SM on every SM
  const int64_t rows = (int64_t)B * Lw;
  const int64_t target_threads = (int64_t)num_sms() * 16 * 32;
  int tpr = 32;
  while (tpr < 256 && rows * tpr < target_threads) tpr *= 2;
  if (tpr == 32) launch_cos<T, VEC, 32>(cur, prev, B, Lw, D, rs, bs, cos_out, stream);
  else if (tpr == 64) launch_cos<T, VEC, 64>(cur, prev, B, Lw, D, rs, bs, cos_out, stream);
  else if (tpr == 128) launch_cos<T, VEC, 128>(cur, prev, B, Lw, D, rs, bs, cos_out, stream);
  else launch_cos<T, VEC, 256>(cur, prev, B, Lw, D, rs, bs, cos_out, stream);
}

template <typename T>
cudaError_t launch_typed(const T* cur, const T* prev, int B, int Lw, int D, int64_t rs,
                         int64_t bs, float* cos_out, cudaStream_t stream) {
  constexpr int E = 16 / sizeof(T);
  const bool vec = (reinterpret_cast<uintptr_t>(cur) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(prev) % 16 == 0) && (D % E == 0) &&
                   (rs % E == 0) && (bs % E == 0);
  if (vec)
    launch_cos_tpr<T, true>(cur, prev, B, Lw, D, rs, bs, cos_out, stream);
  else
    launch_cos_tpr<T, false>(cur, prev, B, Lw, D, rs, bs, cos_out, stream);
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
  launch_pdl(compact_kernel, B, kCompactThreads, 0, stream, cos_out, locked, Lw, tau, idx_base, idx_out,
                                                    count_out);
  return cudaGetLastError();
}

}  // namespace dllm
