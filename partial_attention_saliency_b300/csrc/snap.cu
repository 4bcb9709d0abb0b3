// Structural snapping of the committed block.
//
// LSP ("Beyond Scattered Acceptance: Fast and Coherent Inference for DLMs via
// Longest Stable Prefixes"), technical summary section 2, step 3: the end of
// the selected block moves to the nearest natural boundary (punctuation,
// newline, code symbol) inside the candidate block, so that nothing is frozen
// half way through a word or sentence.  The tokenizer's boundaries come as a
// flag per vocabulary id; the block [start, start + len) then ends after its
// last boundary token at a position >= start + max(min_len, 1) - 1, and keeps
// its length when there is none.
//
// snap_prefix_kernel  one CTA of 256 threads per batch row: the threads scan
//                     the allowed ends of the block for boundary tokens and
//                     a block maximum picks the last one.
#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kSnapThreads = 256;

__global__ void __launch_bounds__(kSnapThreads)
snap_prefix_kernel(const int32_t* tokens, int L, int V, const uint8_t* delim,
                   const int32_t* start, int32_t* len, int min_len, int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  __shared__ int s_best[kSnapThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = __ldca(start + b);
  const int n = __ldca(len + b);
  if (s < 0 || s > L || n < 0 || n > L - s) {  // uniform over the CTA
    if (tid == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
    return;
  }
  const int lo = s + (min_len > 1 ? min_len : 1) - 1;
  const int32_t* row = tokens + (int64_t)b * L;
  int best = -1;
  for (int p = lo + tid; p < s + n; p += kSnapThreads) {
    const int t = __ldca(row + p);
    if (t < 0 || t >= V) {
      report(dev_status, DLLM_ERR_DEVICE_CHECK);
      continue;
    }
    if (__ldca(delim + t) != 0) best = p;  // p grows: the thread's last boundary
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  if (lane == 0) s_best[warp] = best;
  __syncthreads();
  if (tid == 0) {
    for (int w = 0; w < kSnapThreads / 32; ++w) best = max(best, s_best[w]);
    if (best >= 0) len[b] = best - s + 1;
  }
}

}  // namespace

cudaError_t launch_snap_prefix(const int32_t* tokens, int B, int L, int V, const uint8_t* delim,
                               const int32_t* start, int32_t* len, int min_len,
                               int32_t* dev_status, cudaStream_t stream) {
  launch_pdl(snap_prefix_kernel, B, kSnapThreads, 0, stream, tokens, L, V, delim, start, len,
             min_len, dev_status);
  return cudaGetLastError();
}

}  // namespace dllm
