// Longest stable prefix of the remaining active suffix.
//
// LSP ("Beyond Scattered Acceptance: Fast and Coherent Inference for DLMs via
// Longest Stable Prefixes"), technical summary section 2: commit the longest
// contiguous stable block at the head of the remaining active sequence in one
// step, judged by a per-position stability score (step 1); step 4: commit at
// least one token when none is stable.
//
// One CTA per batch row: every thread tests a strided set of the positions
// at and after start (all loads independent, so the scan costs one memory
// round trip instead of one per 32 positions) and keeps the lowest unstable
// position it saw; a block-wide minimum gives the end of the run.  Reads 4
// bytes per scanned position.
#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kPrefixThreads = 256;
constexpr int kPrefixUnroll = 4;

__global__ void __launch_bounds__(kPrefixThreads)
stable_prefix_kernel(const float* score, int L, int32_t* start,
                     float tau, int min_commit, int advance, int32_t* len_out,
                     int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  __shared__ int warp_min[kPrefixThreads / 32];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = __ldca(start + b);
  if (s < 0 || s > L) {
    if (tid == 0) {
      report(dev_status, DLLM_ERR_DEVICE_CHECK);
      len_out[b] = 0;
    }
    return;
  }
  const float* row = score + (int64_t)b * L;
  int first = L;  // lowest unstable position seen by this thread
  for (int base = s; base < L && first == L; base += kPrefixThreads * kPrefixUnroll) {
    float v[kPrefixUnroll];
#pragma unroll
    for (int u = 0; u < kPrefixUnroll; ++u) {
      const int p = base + u * kPrefixThreads + tid;
      v[u] = p < L ? __ldca(row + p) : INFINITY;
    }
#pragma unroll
    for (int u = kPrefixUnroll - 1; u >= 0; --u) {
      const int p = base + u * kPrefixThreads + tid;
      if (p < L && !(v[u] >= tau)) first = p;  // NaN is unstable
    }
  }
  first = warp_min_int(first);
  if (lane == 0) warp_min[warp] = first;
  __syncthreads();
  if (tid == 0) {
    int m = warp_min[0];
#pragma unroll
    for (int w = 1; w < kPrefixThreads / 32; ++w) m = min(m, warp_min[w]);
    int k = m - s;
    if (min_commit && k == 0 && s < L) k = 1;
    len_out[b] = k;
    if (advance) start[b] = s + k;
  }
}

}  // namespace

cudaError_t launch_stable_prefix(const float* score, int B, int L, int32_t* start, float tau,
                                 int min_commit, int advance_start, int32_t* len_out,
                                 int32_t* dev_status, cudaStream_t stream) {
  launch_pdl(stable_prefix_kernel, B, kPrefixThreads, 0, stream, score, L, start, tau, min_commit,
                                                         advance_start, len_out, dev_status);
  return cudaGetLastError();
}

}  // namespace dllm
