// Longest stable prefix of the remaining active suffix.
//
// LSP ("Beyond Scattered Acceptance: Fast and Coherent Inference for DLMs via
// Longest Stable Prefixes"), technical summary section 2: commit the longest
// contiguous stable block at the head of the remaining active sequence in one
// step, judged by a per-position stability score (step 1); step 4: commit at
// least one token when none is stable.
//
// One warp per batch row: 32 positions per ballot, the first zero bit of the
// ballot ends the run.  Reads 4 bytes per scanned position.
#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

__global__ void stable_prefix_kernel(const float* __restrict__ score, int B, int L,
                                     int32_t* __restrict__ start, float tau, int min_commit,
                                     int advance, int32_t* __restrict__ len_out,
                                     int32_t* dev_status) {
  const int b = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const int s = start[b];
  if (s < 0 || s > L) {
    if (lane == 0) {
      report(dev_status, DLLM_ERR_DEVICE_CHECK);
      len_out[b] = 0;
    }
    return;
  }
  const float* row = score + (int64_t)b * L;
  int k = 0;
  for (int base = s; base < L; base += 32) {
    const int p = base + lane;
    const bool stable = p < L && row[p] >= tau;  // NaN and past-the-end are unstable
    const unsigned ball = __ballot_sync(0xffffffffu, stable);
    if (ball == 0xffffffffu) {
      k += 32;
      continue;
    }
    k += __ffs(~ball) - 1;
    break;
  }
  if (min_commit && k == 0 && s < L) k = 1;
  __syncwarp();
  if (lane == 0) {
    len_out[b] = k;
    if (advance) start[b] = s + k;
  }
}

}  // namespace

cudaError_t launch_stable_prefix(const float* score, int B, int L, int32_t* start, float tau,
                                 int min_commit, int advance_start, int32_t* len_out,
                                 int32_t* dev_status, cudaStream_t stream) {
  const int threads = 128;
  const int64_t total = (int64_t)B * 32;
  const unsigned grid = (unsigned)((total + threads - 1) / threads);
  stable_prefix_kernel<<<grid, threads, 0, stream>>>(score, B, L, start, tau, min_commit,
                                                     advance_start, len_out, dev_status);
  return cudaGetLastError();
}

}  // namespace dllm
