// KV-cache update: fresh K/V rows of the active positions into the cache.
//
// SureLock ("Stopping Computation for Converged Tokens in Masked Diffusion-LM
// Decoding"), technical summary section 2: K/V of locked positions stay
// cached and other tokens attend to them; only active positions get new K/V.
// LSP, technical summary section 2 ("KV Cache"): contiguous appends -- a run
// of consecutive indices is simply consecutive rows here.
//
// CTAs of batch row b take its active rows round-robin; a row (H*d elements
// of K and of V) is contiguous in both the new-row buffer and the cache, so
// the copy is a pair of coalesced 16-byte streams.  HBM bound: 4 * H * d * sizeof(T) bytes per
// active row (read K/V new, write K/V cache).
#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kScatterThreads = 256;

template <bool VEC>
__global__ void __launch_bounds__(kScatterThreads)
kv_scatter_kernel(char* kc, char* vc, const char* kn,
                  const char* vn, int L, int M_max, int64_t row_bytes,
                  const int32_t* idx, const int32_t* count,
                  int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  const int b = blockIdx.y;
  int n = __ldca(count + b);
  if (n < 0 || n > M_max) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
    n = n < 0 ? 0 : M_max;
  }
  const int32_t* ib = idx + (int64_t)b * M_max;
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const int p = __ldca(ib + i);
    const bool ordered = (i == 0) || (__ldca(ib + i - 1) < p);
    if (p < 0 || p >= L || !ordered) {
      if (threadIdx.x == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
      continue;
    }
    const int64_t src = ((int64_t)b * M_max + i) * row_bytes;
    const int64_t dst = ((int64_t)b * L + p) * row_bytes;
    if constexpr (VEC) {
      const int64_t nv = row_bytes / 16;
      const uint4* sk = reinterpret_cast<const uint4*>(kn + src);
      const uint4* sv = reinterpret_cast<const uint4*>(vn + src);
      uint4* dk = reinterpret_cast<uint4*>(kc + dst);
      uint4* dv = reinterpret_cast<uint4*>(vc + dst);
      for (int64_t base = 0; base < nv; base += 2 * kScatterThreads) {
        uint4 a[2], c[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int64_t v = base + u * kScatterThreads + threadIdx.x;
          if (v < nv) {
            a[u] = ld_stream16(sk + v);
            c[u] = ld_stream16(sv + v);
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int64_t v = base + u * kScatterThreads + threadIdx.x;
          if (v < nv) {
            dk[v] = a[u];
            dv[v] = c[u];
          }
        }
      }
    } else {
      for (int64_t k = threadIdx.x; k < row_bytes; k += kScatterThreads) {
        kc[dst + k] = kn[src + k];
        vc[dst + k] = vn[src + k];
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_scatter(void* k_cache, void* v_cache, const void* k_new,
                              const void* v_new, int dtype, int B, int L, int H, int d,
                              int M_max, const int32_t* idx, const int32_t* count,
                              int32_t* dev_status, cudaStream_t stream) {
  const int64_t elt = dtype == DLLM_BF16 ? 2 : 4;
  const int64_t row_bytes = (int64_t)H * d * elt;
  const bool vec = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(k_cache) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(v_cache) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(k_new) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(v_new) % 16 == 0;
  // rows are dealt round-robin to at most ~8 resident CTAs per SM over all
  // batch rows; CTAs past a batch row's count exit after reading it
  const int per_b = (8 * num_sms() + B - 1) / B;
  dim3 grid(M_max < per_b ? M_max : per_b, B);
  if (vec)
    launch_pdl(kv_scatter_kernel<true>, grid, kScatterThreads, 0, stream,
        static_cast<char*>(k_cache), static_cast<char*>(v_cache),
        static_cast<const char*>(k_new), static_cast<const char*>(v_new), L, M_max, row_bytes,
        idx, count, dev_status);
  else
    launch_pdl(kv_scatter_kernel<false>, grid, kScatterThreads, 0, stream,
        static_cast<char*>(k_cache), static_cast<char*>(v_cache),
        static_cast<const char*>(k_new), static_cast<const char*>(v_new), L, M_max, row_bytes,
        idx, count, dev_status);
  return cudaGetLastError();
}

}  // namespace dllm
