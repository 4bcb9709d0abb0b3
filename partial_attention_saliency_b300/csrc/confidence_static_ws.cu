// dllm_confidence_static_ws: the confidence entry point for callers that
// cannot allocate device memory (for instance a plugin handed only raw input
// and output pointers by its host framework, or a latency-critical caller that
// cannot afford cudaMalloc's device-wide synchronisation).
//
// The split-row confidence kernels need scratch for their per-chunk partial
// results.  Here that scratch is a file-scope device array of a fixed size,
// created when the library's module is loaded on a device and held until the
// process exits.  In host code `g_confidence_scratch` only names a host-side
// stand-in, so its device address is looked up with cudaGetSymbolAddress,
// once per device, with that device current, and that address is what the
// kernels receive.  Calls share the array and leave their partials in it;
// calls that overlap on the GPU race on it.
#include <cstdio>
#include <mutex>

#include "dllm.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = DLLM_CONFIDENCE_STATIC_WS_BYTES;
__device__ __align__(256) unsigned char g_confidence_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call for that device).
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_confidence_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" dllm_status dllm_confidence_static_ws(
    const void* logits, int dtype, int B, int R_src, int V, int64_t row_stride,
    int64_t batch_stride, int R_max, const int32_t* row_idx, const int32_t* count,
    const int32_t* out_idx, int out_cols, float* conf_out, int32_t* argmax_out,
    float* margin_out, int32_t* dev_status, void* stream) {
  // The cheap argument checks first, so that a rejected call returns before
  // it touches the CUDA runtime (dllm_confidence repeats them all).
  if (logits == nullptr || conf_out == nullptr || argmax_out == nullptr ||
      (dtype != DLLM_F32 && dtype != DLLM_BF16) || B < 1 || R_src < 1 || R_max < 1 || V < 2 ||
      out_cols < 1)
    return (dllm_status)dllm::set_last_error(
        DLLM_ERR_INVALID_ARG, "dllm_confidence_static_ws: NULL pointer, dtype or size out of range");
  const size_t need = dllm_confidence_workspace_bytes(B, R_max, V, dtype);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "dllm_confidence_static_ws: B*R_max=%lld rows of V=%d need %zu scratch bytes, "
             "above the static maximum of %zu bytes",
             (long long)B * R_max, V, need, kScratchBytes);
    return (dllm_status)dllm::set_last_error(DLLM_ERR_INVALID_ARG, msg);
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "dllm_confidence_static_ws: scratch address lookup failed: %s",
             cudaGetErrorString(e));
    return (dllm_status)dllm::set_last_error(DLLM_ERR_CUDA, msg);
  }
  return dllm_confidence(logits, dtype, B, R_src, V, row_stride, batch_stride, R_max, row_idx,
                         count, out_idx, out_cols, conf_out, argmax_out, margin_out, scratch,
                         kScratchBytes, dev_status, stream);
}
