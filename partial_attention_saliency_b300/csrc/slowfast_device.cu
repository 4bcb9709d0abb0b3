// SlowFast sampling on the device: the phase controller and the tokens each
// phase unmasks, so that a decoding loop never reads a prediction back to
// the host.
//
// SlowFast ("Accelerating Diffusion Large Language Models with SlowFast
// Sampling: The Three Golden Principles"), section 2 (pipeline): the slow,
// exploratory phase selects the most confident tokens of an exploration
// window while the prediction of the convergence point e_cand is watched over
// a sliding window of steps; once its variance falls below sigma^2_stable the
// region [s_cycle, e_cycle] is stable, and the fast phase unmasks every
// masked token of the region whose confidence exceeds tau_high_conf at once.
//
// slowfast_observe_kernel  one thread per batch row: the controller of the
//                          host-side dllm_slowfast_observe, its predictions
//                          held in a device state array.
// slowfast_select_kernel   one CTA of 1024 threads per batch row: the fast
//                          phase compacts the passing positions of its
//                          region in ascending order; the slow phase takes
//                          the k best (confidence descending, position
//                          ascending) of its window by k block-wide minimum
//                          rounds over 64-bit keys, then compacts them in
//                          ascending order.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kSfThreads = 1024;
constexpr int kSfPerThread = 16;  // window positions per thread (slow phase)

// Predictions of the current cycle per batch row: state[b * (W + 1)] holds
// how many (0 .. W), followed by them, oldest first.
__global__ void slowfast_observe_kernel(int32_t* state, int B, int W, double sigma2,
                                        const int32_t* start, const int32_t* pred_len,
                                        int32_t* phase_out, int32_t* region_end_out,
                                        int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int32_t* s = state + (int64_t)b * (W + 1);
  int n = s[0];
  if (n < 0 || n > W) {  // not a state this kernel wrote: start the cycle afresh
    report(dev_status, DLLM_ERR_DEVICE_CHECK);
    n = 0;
  }
  const int64_t st = __ldca(start + b);
  const int64_t e = st + __ldca(pred_len + b);
  if (n == W) {  // the oldest prediction leaves the window
    for (int i = 1; i < W; ++i) s[i] = s[i + 1];
    n = W - 1;
  }
  s[1 + n] = (int32_t)e;
  ++n;
  int32_t ph = 0, end = -1;
  if (n == W && e > st) {
    int64_t s1 = 0, s2 = 0;
    for (int i = 1; i <= W; ++i) {
      const int64_t x = s[i];
      s1 += x;
      s2 += x * x;
    }
    const int64_t num = (int64_t)W * s2 - s1 * s1;  // W^2 times the population variance
    if ((double)num < sigma2 * (double)((int64_t)W * W)) {
      ph = 1;
      end = (int32_t)e;
      n = 0;  // a fast step closes the cycle
    }
  }
  s[0] = n;
  phase_out[b] = ph;
  region_end_out[b] = end;
}

// Ascending order = descending confidence, equal confidences by ascending
// position (-0 equals +0); NaN confidences are not candidates.
__device__ __forceinline__ uint64_t rank_key(float c, int pos) {
  if (c == 0.f) c = 0.f;
  const uint32_t u = __float_as_uint(c);
  const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)(~asc) << 32) | (uint32_t)pos;
}

__device__ __forceinline__ uint64_t warp_min_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w < v ? w : v;
  }
  return v;
}

// Block-wide exclusive rank of `flag` in thread order and the block total.
__device__ __forceinline__ int block_rank(bool flag, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) s_warp[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    const int v = s_warp[lane];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int w = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += w;
    }
    s_warp[lane] = incl - v;
    if (lane == 31) s_warp[32] = incl;
  }
  __syncthreads();
  const int r = s_warp[warp] + in_warp;
  *total = s_warp[32];
  __syncthreads();  // s_warp is reused by the next call
  return r;
}

__global__ void __launch_bounds__(kSfThreads)
slowfast_select_kernel(const float* conf, const uint8_t* masked, int L, const int32_t* start,
                       const int32_t* phase, const int32_t* region_end, float tau_high,
                       int width, int k, int32_t* idx_out, int32_t* count_out,
                       int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  __shared__ int s_warp[33];
  __shared__ uint64_t s_min[32];
  const int b = blockIdx.x, t = threadIdx.x;
  const float* c = conf + (int64_t)b * L;
  const uint8_t* m = masked ? masked + (int64_t)b * L : nullptr;
  int32_t* out = idx_out + (int64_t)b * L;
  int st = __ldca(start + b);
  if (st < 0 || st > L) {
    if (t == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
    st = L;  // nothing selected
  }
  const bool fast = __ldca(phase + b) == 1;
  int n = 0;  // positions written so far
  if (fast) {
    int hi = __ldca(region_end + b);
    if (hi < st || hi > L) {
      if (t == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
      hi = hi < st ? st : L;
    }
    for (int base = st; base < hi; base += kSfThreads) {
      const int p = base + t;
      const bool pass = p < hi && (m == nullptr || m[p] != 0) && __ldca(c + p) > tau_high;
      int tot;
      const int r = block_rank(pass, s_warp, &tot);
      if (pass) out[n + r] = p;
      n += tot;
    }
  } else {
    const int hi = (int)min((int64_t)st + width, (int64_t)L);
    uint64_t key[kSfPerThread];
#pragma unroll
    for (int i = 0; i < kSfPerThread; ++i) {
      const int p = st + i * kSfThreads + t;
      key[i] = ~0ull;
      if (p < hi && (m == nullptr || m[p] != 0)) {
        const float v = __ldca(c + p);
        if (!isnan(v)) key[i] = rank_key(v, p);
      }
    }
    uint32_t picked = 0;  // bit i: key[i] selected
    const int lane = t & 31, warp = t >> 5;
    for (int round = 0; round < k; ++round) {
      uint64_t best = ~0ull;
#pragma unroll
      for (int i = 0; i < kSfPerThread; ++i)
        if (!((picked >> i) & 1u) && key[i] < best) best = key[i];
      best = warp_min_u64(best);
      if (lane == 0) s_min[warp] = best;
      __syncthreads();
      best = warp_min_u64(s_min[lane]);
      __syncthreads();  // s_min is rewritten next round
      if (best == ~0ull) break;  // fewer candidates than k
#pragma unroll
      for (int i = 0; i < kSfPerThread; ++i)
        if (key[i] == best) picked |= 1u << i;  // keys are distinct (they hold the position)
    }
    // the picked positions in ascending order: window rows i = 0, 1, ... in turn
    for (int i = 0; i < kSfPerThread; ++i) {
      if (st + i * kSfThreads >= hi) break;  // block-uniform
      const bool pass = (picked >> i) & 1u;
      int tot;
      const int r = block_rank(pass, s_warp, &tot);
      if (pass) out[n + r] = st + i * kSfThreads + t;
      n += tot;
    }
  }
  for (int p = n + t; p < L; p += kSfThreads) out[p] = -1;
  if (t == 0) count_out[b] = n;
}

}  // namespace

int slowfast_select_max_width() { return kSfThreads * kSfPerThread; }

cudaError_t launch_slowfast_observe(int32_t* state, int B, int W, double sigma2,
                                    const int32_t* start, const int32_t* pred_len,
                                    int32_t* phase_out, int32_t* region_end_out,
                                    int32_t* dev_status, cudaStream_t stream) {
  const int threads = 128;
  launch_pdl(slowfast_observe_kernel, (B + threads - 1) / threads, threads, 0, stream, state, B,
             W, sigma2, start, pred_len, phase_out, region_end_out, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_slowfast_select(const float* conf, const uint8_t* masked, int B, int L,
                                   const int32_t* start, const int32_t* phase,
                                   const int32_t* region_end, float tau_high, int width, int k,
                                   int32_t* idx_out, int32_t* count_out, int32_t* dev_status,
                                   cudaStream_t stream) {
  launch_pdl(slowfast_select_kernel, B, kSfThreads, 0, stream, conf, masked, L, start, phase,
             region_end, tau_high, width, k, idx_out, count_out, dev_status);
  return cudaGetLastError();
}

}  // namespace dllm
