// Approximate attention update of the stable rows (the non-salient path).
//
// DyLLM ("DyLLM: Efficient Diffusion LLM Inference via Saliency-based Token
// Selection and Partial Attention"), technical summary, Methodology 2
// (non-salient path): a stable row keeps its attention weights and its output
// moves by the change of the salient tokens' values weighted by them, at cost
// O(N |A_t|).  The weights of the previous step are recovered exactly from
// the cached query, the previous keys of the salient positions and the cached
// log-sum-exp:
//   o_i += sum_{a < count} 2^(log2e (scale q_i . k_{idx_a} - lse_i)) (v_new_a - v_{idx_a}).
//
// approx_update_kernel  one CTA of 256 threads per (64 stable rows, head,
//                       batch row).  The tile's queries (transposed) and
//                       log-sum-exps stay in shared memory; the salient
//                       columns are taken 64 at a time: their previous keys
//                       (transposed) and value changes are gathered into
//                       shared memory, each thread computes a 4 x 4 block of
//                       S and of P, then a 4 x (d/16) block of P dV is added
//                       to its accumulators.  FMA-pipe (SIMT) arithmetic in
//                       float32; float32 inputs and head dims 32 and 64 (bf16
//                       with head dim 128 runs on the tensor cores,
//                       approx_update_tc.cu).
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kAuRows = 64;     // stable rows per CTA
constexpr int kAuCols = 64;     // salient columns per tile
constexpr int kAuThreads = 256;  // 16 x 16 threads
constexpr int kAuPad = 4;       // floats of padding per shared-memory row

template <int D>
struct AuSmem {
  static constexpr int kT = kAuRows + kAuPad;     // row length of the transposed tiles
  static constexpr int kV = D + kAuPad;           // row length of the value-change tile
  static constexpr int kQt = 0;                   // [D][kT] queries, transposed
  static constexpr int kKt = kQt + D * kT;        // [D][kT] keys, transposed
  static constexpr int kVd = kKt + D * kT;        // [kAuCols][kV] value changes
  static constexpr int kPt = kVd + kAuCols * kV;  // [kAuCols][kT] probabilities, transposed
  static constexpr int kLse = kPt + kAuCols * kT;  // [kAuRows] lse * log2(e)
  static constexpr int kFloats = kLse + kAuRows;
  static constexpr int kBytes = kFloats * 4 + 2 * kAuRows * 4;  // + row and column positions
};

template <typename T>
__device__ __forceinline__ float to_f(T x) {
  if constexpr (std::is_same<T, float>::value) {
    return x;
  } else {
    return __bfloat162float(x);
  }
}

template <typename T>
__device__ __forceinline__ T from_f(float x) {
  if constexpr (std::is_same<T, float>::value) {
    return x;
  } else {
    return __float2bfloat16_rn(x);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kAuThreads)
approx_update_kernel(const T* q, const float* lse, const T* k, const T* v, const T* v_new,
                     const int32_t* idx, const int32_t* count, const int32_t* stable_idx,
                     const int32_t* stable_count, T* o, int L, int H, int M_max, int N_max,
                     float scale_log2e, int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  using S = AuSmem<D>;
  constexpr int CPT = D / 16;  // output columns per thread
  extern __shared__ float4 au_smem4[];
  float* sm = reinterpret_cast<float*>(au_smem4);
  float* Qt = sm + S::kQt;
  float* Kt = sm + S::kKt;
  float* Vd = sm + S::kVd;
  float* Pt = sm + S::kPt;
  float* lse_s = sm + S::kLse;
  int* rows_s = reinterpret_cast<int*>(sm + S::kFloats);
  int* cols_s = rows_s + kAuRows;

  const int b = blockIdx.z, h = blockIdx.y, r0 = blockIdx.x * kAuRows;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  int ns = __ldca(stable_count + b);
  int na = __ldca(count + b);
  if (ns < 0 || ns > N_max || na < 0 || na > M_max) {
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
    ns = ns < 0 ? 0 : (ns > N_max ? N_max : ns);
    na = na < 0 ? 0 : (na > M_max ? M_max : na);
  }
  if (r0 >= ns || na == 0) return;  // uniform over the CTA

  // 1. the tile's stable rows, their queries (transposed) and lse
  if (tid < kAuRows) {
    const int i = r0 + tid;
    int pos = -1;
    if (i < ns) {
      pos = __ldca(stable_idx + (int64_t)b * N_max + i);
      if (pos < 0 || pos >= L) {
        if (h == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
        pos = -1;
      }
    }
    rows_s[tid] = pos;
    lse_s[tid] = pos >= 0 ? __ldca(lse + ((int64_t)b * H + h) * L + pos) * kLog2e : 0.f;
  }
  __syncthreads();
  for (int e = tid; e < kAuRows * D; e += kAuThreads) {
    const int r = e / D, kk = e - r * D;
    const int pos = rows_s[r];
    Qt[kk * S::kT + r] = pos >= 0 ? to_f(q[(((int64_t)b * L + pos) * H + h) * D + kk]) : 0.f;
  }

  float acc[4][CPT];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < CPT; ++j) acc[r][j] = 0.f;

  for (int a0 = 0; a0 < na; a0 += kAuCols) {
    // 2. the salient columns of this tile: previous keys and value changes
    if (tid < kAuCols) {
      const int a = a0 + tid;
      int pos = -1;
      if (a < na) {
        pos = __ldca(idx + (int64_t)b * M_max + a);
        if (pos < 0 || pos >= L) {
          if (h == 0 && blockIdx.x == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
          pos = -1;
        }
      }
      cols_s[tid] = pos;
    }
    __syncthreads();  // also orders the Qt stores before the first use
    for (int e = tid; e < kAuCols * D; e += kAuThreads) {
      const int c = e / D, kk = e - c * D;
      const int pos = cols_s[c];
      float kv = 0.f, dv = 0.f;
      if (pos >= 0) {
        const int64_t src = (((int64_t)b * L + pos) * H + h) * D + kk;
        kv = to_f(k[src]);
        dv = to_f(v_new[(((int64_t)b * M_max + a0 + c) * H + h) * D + kk]) - to_f(v[src]);
      }
      Kt[kk * S::kT + c] = kv;
      Vd[c * S::kV + kk] = dv;
    }
    __syncthreads();
    // 3. S = Q K^T for rows ty*4 .. +3 and columns tx*4 .. +3, then P
    float s[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[r][c] = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < D; ++kk) {
      const float4 qv = *reinterpret_cast<const float4*>(Qt + kk * S::kT + ty * 4);
      const float4 kv = *reinterpret_cast<const float4*>(Kt + kk * S::kT + tx * 4);
      const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
      const float ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[r][c] = fmaf(qa[r], ka[c], s[r][c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const bool col_ok = cols_s[tx * 4 + c] >= 0;
      float pr[4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
        pr[r] = col_ok ? ex2_approx(fmaf(s[r][c], scale_log2e, -lse_s[ty * 4 + r])) : 0.f;
      *reinterpret_cast<float4*>(Pt + (tx * 4 + c) * S::kT + ty * 4) =
          make_float4(pr[0], pr[1], pr[2], pr[3]);
    }
    __syncthreads();
    // 4. dO += P dV for rows ty*4 .. +3 and columns tx*CPT .. +CPT-1
    const int cmax = min(kAuCols, na - a0);
    for (int c = 0; c < cmax; ++c) {
      const float4 pv = *reinterpret_cast<const float4*>(Pt + c * S::kT + ty * 4);
      const float pa[4] = {pv.x, pv.y, pv.z, pv.w};
      float dv[CPT];
      const float* vrow = Vd + c * S::kV + tx * CPT;
      if constexpr (CPT % 4 == 0) {
#pragma unroll
        for (int j = 0; j < CPT; j += 4) {
          const float4 t = *reinterpret_cast<const float4*>(vrow + j);
          dv[j] = t.x;
          dv[j + 1] = t.y;
          dv[j + 2] = t.z;
          dv[j + 3] = t.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < CPT; j += 2) {
          const float2 t = *reinterpret_cast<const float2*>(vrow + j);
          dv[j] = t.x;
          dv[j + 1] = t.y;
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[r][j] = fmaf(pa[r], dv[j], acc[r][j]);
    }
    __syncthreads();  // the next tile overwrites cols_s, Kt, Vd and Pt
  }

  // 5. o += dO on the stable rows
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int pos = rows_s[ty * 4 + r];
    if (pos < 0) continue;
    T* orow = o + (((int64_t)b * L + pos) * H + h) * D + tx * CPT;
#pragma unroll
    for (int j = 0; j < CPT; ++j) orow[j] = from_f<T>(to_f(orow[j]) + acc[r][j]);
  }
}

template <typename T, int D>
cudaError_t launch_au(const void* q, const float* lse, const void* k, const void* v,
                      const void* v_new, int B, int L, int H, int M_max, const int32_t* idx,
                      const int32_t* count, int N_max, const int32_t* stable_idx,
                      const int32_t* stable_count, float scale, void* o, int32_t* dev_status,
                      cudaStream_t stream) {
  constexpr int bytes = AuSmem<D>::kBytes;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(approx_update_kernel<T, D>),
                                    bytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((N_max + kAuRows - 1) / kAuRows), (unsigned)H, (unsigned)B);
  launch_pdl(approx_update_kernel<T, D>, grid, kAuThreads, (size_t)bytes, stream,
             static_cast<const T*>(q), lse, static_cast<const T*>(k), static_cast<const T*>(v),
             static_cast<const T*>(v_new), idx, count, stable_idx, stable_count,
             static_cast<T*>(o), L, H, M_max, N_max, scale * kLog2e, dev_status);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_au_d(int d, const void* q, const float* lse, const void* k, const void* v,
                        const void* v_new, int B, int L, int H, int M_max, const int32_t* idx,
                        const int32_t* count, int N_max, const int32_t* stable_idx,
                        const int32_t* stable_count, float scale, void* o, int32_t* dev_status,
                        cudaStream_t stream) {
  switch (d) {
    case 32:
      return launch_au<T, 32>(q, lse, k, v, v_new, B, L, H, M_max, idx, count, N_max, stable_idx,
                              stable_count, scale, o, dev_status, stream);
    case 64:
      return launch_au<T, 64>(q, lse, k, v, v_new, B, L, H, M_max, idx, count, N_max, stable_idx,
                              stable_count, scale, o, dev_status, stream);
    case 128:
      return launch_au<T, 128>(q, lse, k, v, v_new, B, L, H, M_max, idx, count, N_max,
                               stable_idx, stable_count, scale, o, dev_status, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_approx_attention_update(const void* q, const float* lse, const void* k,
                                           const void* v, const void* v_new, int dtype, int B,
                                           int L, int H, int d, int M_max, const int32_t* idx,
                                           const int32_t* count, int N_max,
                                           const int32_t* stable_idx,
                                           const int32_t* stable_count, float scale, void* o,
                                           int32_t* dev_status, cudaStream_t stream) {
  // bf16 with head dim 128: the tensor-core kernel (approx_update_tc.cu)
  if (approx_update_tc_supported(dtype, d, q, k, v, v_new, o))
    return launch_approx_update_tc(q, lse, k, v, v_new, B, L, H, M_max, idx, count, N_max,
                                   stable_idx, stable_count, scale, o, dev_status, stream);
  if (dtype == DLLM_BF16)
    return launch_au_d<__nv_bfloat16>(d, q, lse, k, v, v_new, B, L, H, M_max, idx, count, N_max,
                                      stable_idx, stable_count, scale, o, dev_status, stream);
  return launch_au_d<float>(d, q, lse, k, v, v_new, B, L, H, M_max, idx, count, N_max,
                            stable_idx, stable_count, scale, o, dev_status, stream);
}

}  // namespace dllm
