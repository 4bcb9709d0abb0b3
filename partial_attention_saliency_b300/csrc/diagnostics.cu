// Diagnostics entry points: checks of the library's own machinery that the
// step's calls do not expose.
//
// dllm_exp2_fma_eval       the FMA-pipe 2^x (Cody-Waite split and the degree-4
//                          polynomial of fit_exp2_poly.py) that the attention
//                          kernels use for part of their exponentials, on an
//                          array, so that its error bound can be checked
//                          against a float64 reference.
// dllm_set_wait_limit      the number of clock cycles after which the bounded
//                          pipeline waits of the streaming confidence kernel
//                          and the attention forward kernel give up, so that
//                          a test can make a wait run out and check that the
//                          kernel records DLLM_ERR_TIMEOUT, drains its copies
//                          and returns.  Drains always keep the long limit.
// dllm_read_stream         the read-streaming reference of a single launch:
//                          one persistent CTA per SM copies a buffer into a
//                          four-stage shared-memory ring with cp.async.bulk
//                          and does nothing else, so its time for a given
//                          byte count is what one launch of a memory-bound
//                          kernel of that size can reach on this GPU (launch,
//                          ramp-up and tail included).
#include <atomic>

#include "common.cuh"
#include "dllm.h"
#include "internal.h"
#include "sm100.cuh"

namespace dllm {
namespace {

std::atomic<long long> g_wait_limit{sm100::kWaitLimitDefault};

__global__ void exp2_fma_eval_kernel(const float* x, float* y, int n) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float2 a = make_float2(x[i], i + 1 < n ? x[i + 1] : 0.f);
  const float2 r = exp2_poly2(a);
  y[i] = r.x;
  if (i + 1 < n) y[i + 1] = r.y;
}

constexpr int kRsStages = 4;
constexpr uint32_t kRsChunk = 32768;
constexpr uint32_t kRsSmem = kRsStages * kRsChunk + 1024;

// Thread 0 streams the CTA's chunks (c = blockIdx.x, + gridDim.x, ...) into
// the ring; thread 32 waits for each, adds its byte at offset 16 * (g % 16)
// (g: the chunk's rank in the CTA's sequence; offset 0 when the chunk is
// shorter) into the checksum and frees the stage.
__global__ void __launch_bounds__(64, 1)
read_stream_kernel(const uint8_t* buf, int64_t bytes, uint32_t* sink, int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  __shared__ uint64_t full[kRsStages], empty[kRsStages];
  __shared__ int abort_s;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRsStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    abort_s = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort = &abort_s;
  const int64_t nch = (bytes + kRsChunk - 1) / kRsChunk;
  if (threadIdx.x == 0) {
    int g = 0;
    for (int64_t c = blockIdx.x; c < nch; c += gridDim.x, ++g) {
      const int s = g % kRsStages;
      if (g >= kRsStages && !mbar_wait(&empty[s], ((g / kRsStages) - 1) & 1, abort)) break;
      const int64_t off = c * kRsChunk;
      const uint32_t n = (uint32_t)(bytes - off < (int64_t)kRsChunk ? bytes - off : kRsChunk);
      mbar_expect_tx(&full[s], n);
      bulk_load(ring + (size_t)s * kRsChunk, buf + off, n, &full[s]);
    }
    int none = 0;  // never leave with copies in flight
    for (int k = g - kRsStages < 0 ? 0 : g - kRsStages; k < g; ++k)
      mbar_wait(&full[k % kRsStages], (k / kRsStages) & 1, &none);
    if (none || *abort) report(dev_status, DLLM_ERR_TIMEOUT);
  } else if (threadIdx.x == 32) {
    uint32_t acc = 0;
    int g = 0;
    for (int64_t c = blockIdx.x; c < nch; c += gridDim.x, ++g) {
      const int s = g % kRsStages;
      if (!mbar_wait(&full[s], (g / kRsStages) & 1, abort)) break;
      const int64_t n = bytes - c * kRsChunk;  // this chunk's size (the last may be short)
      const uint32_t o = (int64_t)((g & 15) * 16) < n ? (uint32_t)(g & 15) * 16u : 0u;
      acc += ring[(size_t)s * kRsChunk + o];
      mbar_arrive(&empty[s]);
    }
    atomicAdd(sink, acc);
  }
}

}  // namespace

long long wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

}  // namespace dllm

extern "C" dllm_status dllm_exp2_fma_eval(const float* x, float* y, int n, void* stream) {
  if (x == nullptr || y == nullptr || n < 1)
    return (dllm_status)dllm::set_last_error(DLLM_ERR_INVALID_ARG,
                                             "dllm_exp2_fma_eval: NULL pointer or n < 1");
  const int threads = 256;
  const int pairs = (n + 1) / 2;
  dllm::launch_pdl(dllm::exp2_fma_eval_kernel, (pairs + threads - 1) / threads, threads, 0,
                   static_cast<cudaStream_t>(stream), x, y, n);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return (dllm_status)dllm::set_last_error(DLLM_ERR_CUDA, cudaGetErrorString(e));
  return DLLM_OK;
}

extern "C" dllm_status dllm_set_wait_limit(long long cycles) {
  if (cycles < 0)
    return (dllm_status)dllm::set_last_error(DLLM_ERR_INVALID_ARG,
                                             "dllm_set_wait_limit: negative cycle count");
  dllm::g_wait_limit.store(cycles == 0 ? dllm::sm100::kWaitLimitDefault : cycles,
                           std::memory_order_relaxed);
  return DLLM_OK;
}

extern "C" dllm_status dllm_read_stream(const void* buf, size_t bytes, uint32_t* sink,
                                        int32_t* dev_status, void* stream) {
  if (buf == nullptr || sink == nullptr || dev_status == nullptr || bytes < 16 ||
      bytes % 16 != 0 || reinterpret_cast<uintptr_t>(buf) % 16 != 0)
    return (dllm_status)dllm::set_last_error(
        DLLM_ERR_INVALID_ARG,
        "dllm_read_stream: NULL pointer, or bytes not a positive multiple of 16, or buf not "
        "16-byte aligned");
  cudaError_t e = dllm::ensure_smem_limit(reinterpret_cast<const void*>(dllm::read_stream_kernel),
                                          (int)dllm::kRsSmem);
  if (e == cudaSuccess) {
    dllm::launch_pdl(dllm::read_stream_kernel, dllm::num_sms(), 64, dllm::kRsSmem,
                     static_cast<cudaStream_t>(stream), static_cast<const uint8_t*>(buf),
                     (int64_t)bytes, sink, dev_status);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess)
    return (dllm_status)dllm::set_last_error(DLLM_ERR_CUDA, cudaGetErrorString(e));
  return DLLM_OK;
}
