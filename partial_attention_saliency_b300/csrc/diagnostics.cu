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
