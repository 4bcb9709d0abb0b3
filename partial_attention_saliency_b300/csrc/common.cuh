// Device helpers shared by the kernels of libdllm (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "dllm.h"

namespace dllm {

constexpr float kLog2e = 1.4426950408889634f;

// First device-side error wins; the kernel then skips the offending work item.
__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// bfloat16 halves of a 32-bit word, widened to float32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 16-byte streaming load that does not allocate in L1.  A coherent load,
// never the non-coherent (ld.global.nc) path: with programmatic dependent
// launch a kernel is resident while the previous kernel still runs, so no
// buffer is read-only for a whole kernel lifetime, which .nc requires.  For
// the same reason no kernel parameter of this library is __restrict__ and
// scalar reads of buffers other kernels write use __ldca (coherent).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Hardware base-2 exponential (MUFU.EX2), flush-to-zero approximation.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x for a pair on the FMA pipe (x <= 128): Cody-Waite split x = n + f with
// n = round(x) (the 1.5 * 2^23 shifter), f in [-1/2, 1/2]; 2^f from a degree-4
// polynomial (relative-error minimax fit of 2^f on [-1/2, 1/2] by Lawson's
// iteratively reweighted least squares: fit_exp2_poly.py in this directory
// prints these coefficients; max relative error 2.64e-6 for the polynomial,
// 2.7e-6 for the whole evaluation in float32); 2^n added to the exponent
// field.  x is clamped at -125, so arguments below it give 2^-125 (about
// 2e-38) instead of 0.
__device__ __forceinline__ float2 exp2_poly2(float2 x) {
  x.x = fmaxf(x.x, -125.0f);
  x.y = fmaxf(x.y, -125.0f);
  const float2 shifter = make_float2(12582912.0f, 12582912.0f);
  const float2 t = __fadd2_rn(x, shifter);
  const float2 n = __fadd2_rn(t, make_float2(-12582912.0f, -12582912.0f));
  const float2 f = __fadd2_rn(x, make_float2(-n.x, -n.y));
  float2 p = make_float2(0x1.3997d6p-7f, 0x1.3997d6p-7f);
  p = __ffma2_rn(p, f, make_float2(0x1.ca144p-5f, 0x1.ca144p-5f));
  p = __ffma2_rn(p, f, make_float2(0x1.ec06dap-3f, 0x1.ec06dap-3f));
  p = __ffma2_rn(p, f, make_float2(0x1.62e0dcp-1f, 0x1.62e0dcp-1f));
  p = __ffma2_rn(p, f, make_float2(0x1.ffffe8p-1f, 0x1.ffffe8p-1f));
  return make_float2(__uint_as_float(__float_as_uint(p.x) + (__float_as_uint(t.x) << 23)),
                     __uint_as_float(__float_as_uint(p.y) + (__float_as_uint(t.y) << 23)));
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization (launch_pdl below): its CTAs may
// become resident while the previous kernel on the stream is still running,
// and pdl_wait() blocks until that kernel has completed and its memory
// operations are visible.  Each kernel calls pdl_wait() before its first
// global read or write, so the ordering of the stream is unchanged; it then
// calls pdl_trigger() to let the next kernel's CTAs launch early.  Without
// the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same launch without programmatic stream serialization: the kernel's
// CTAs become resident only once the previous kernel on the stream has
// completed (its pdl_wait() then returns at once).
template <typename... KArgs, typename... Args>
cudaError_t launch_serial(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f32(float x) { return x; }
  static __device__ __forceinline__ float from_f32(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace dllm
