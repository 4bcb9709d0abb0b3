// Confidence (max softmax probability), argmax and logit margin per row.
//
// SlowFast ("Accelerating Diffusion LLMs with SlowFast Sampling"), section 2:
// certainty principle; SureLock, technical summary section 2, locking
// criterion 2: uncertainty 1 - max_v p(v); LSP, technical summary section 2,
// step 1: logit margin = top-1 minus top-2 logit.
//
// conf = 1 / sum_j exp(z_j - m) with m = max_j z_j; argmax = lowest j with
// z_j = m; margin = m - max_{j != argmax} z_j.
//
// Split-row design (HBM bound, V * sizeof(T) bytes per row): a row of
// V = 126464 bf16 logits is 253 KB, and a step scores only a few hundred rows,
// so one CTA per row leaves SMs idle.  conf_partial_kernel gives each CTA one
// 32 KB chunk of one row, loaded in a single burst of 16-byte vectors (8 per
// thread in flight), reduces it to (max, second max, sum exp(z - max),
// argmax) and stores that partial in the workspace; conf_merge_kernel folds
// the partials of each row in a fixed order (deterministic) and writes the
// outputs.  Aligned rows take the streaming kernel below instead of
// conf_partial_kernel.
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace dllm {
namespace {

constexpr int kConfThreads = 256;
constexpr int kConfU = 8;  // 16-byte vectors per thread per chunk

struct ConfPartial {
  float m1;   // maximum
  float m2;   // second largest value (equal to m1 on a tie)
  float l;    // sum of exp(z - m1)
  int arg;    // lowest index reaching m1
};

template <typename T> __host__ __device__ constexpr int vec_elems() { return 16 / (int)sizeof(T); }

template <typename T> __host__ __device__ inline int conf_chunk_elems() {
  return kConfThreads * kConfU * vec_elems<T>();
}

__device__ __forceinline__ ConfPartial merge(const ConfPartial& a, const ConfPartial& b) {
  if (b.m1 == -INFINITY) return a;
  if (a.m1 == -INFINITY) return b;
  ConfPartial r;
  r.m1 = fmaxf(a.m1, b.m1);
  r.l = a.l * ex2_approx((a.m1 - r.m1) * kLog2e) + b.l * ex2_approx((b.m1 - r.m1) * kLog2e);
  if (a.m1 > b.m1) {
    r.arg = a.arg;
    r.m2 = fmaxf(a.m2, b.m1);
  } else if (b.m1 > a.m1) {
    r.arg = b.arg;
    r.m2 = fmaxf(b.m2, a.m1);
  } else {
    r.arg = min(a.arg, b.arg);
    r.m2 = a.m1;
  }
  return r;
}

// Element e of a 16-byte vector, as float32.
template <typename T>
__device__ __forceinline__ float elem_of(const uint4& v, int e) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (std::is_same<T, float>::value) {
    return __uint_as_float(w[e]);
  } else {
    return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
  }
}

// Vector vi of a row: a 16-byte load when it lies inside [0, V) and VEC holds,
// else element-wise loads with -inf past the end of the row.
template <typename T, bool VEC>
__device__ __forceinline__ uint4 load_vec(const T* row, int vi, int V) {
  constexpr int E = vec_elems<T>();
  if (VEC && (vi + 1) * E <= V) return ld_stream16(row + (int64_t)vi * E);
  uint32_t w[4];
  if constexpr (std::is_same<T, float>::value) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = vi * E + k;
      w[k] = i < V ? __float_as_uint(row[i]) : 0xff800000u;
    }
  } else {
    const uint16_t* h = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i0 = vi * E + 2 * k, i1 = i0 + 1;
      const uint32_t lo = i0 < V ? h[i0] : 0xff80u;
      const uint32_t hi = i1 < V ? h[i1] : 0xff80u;
      w[k] = lo | (hi << 16);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ bool row_valid(int b, int r, int R_max, int R_src,
                                          const int32_t* row_idx, const int32_t* count,
                                          int* row_out, bool* bad) {
  int n = count ? __ldca(count + b) : R_max;
  *bad = false;
  if (n < 0 || n > R_max) {
    *bad = true;
    n = n < 0 ? 0 : R_max;
  }
  if (r >= n) return false;
  const int row = row_idx ? __ldca(row_idx + (int64_t)b * R_max + r) : r;
  if (row < 0 || row >= R_src) {
    *bad = true;
    return false;
  }
  *row_out = row;
  return true;
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kConfThreads)
conf_partial_kernel(const T* logits, int R_src, int V, int64_t rs, int64_t bs,
                    int R_max, const int32_t* row_idx,
                    const int32_t* count, int nchunks,
                    ConfPartial* ws) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  constexpr int E = vec_elems<T>();
  const int br = blockIdx.x;
  const int chunk = blockIdx.y;
  const int b = br / R_max, r = br - b * R_max;
  int row;
  bool bad;
  if (!row_valid(b, r, R_max, R_src, row_idx, count, &row, &bad)) return;
  const T* p = logits + (int64_t)b * bs + (int64_t)row * rs;
  const int tid = threadIdx.x;
  const int vbase = chunk * (kConfThreads * kConfU);
  const int nvec = (V + E - 1) / E;

  uint4 v[kConfU];
#pragma unroll
  for (int u = 0; u < kConfU; ++u) {
    const int vi = vbase + u * kConfThreads + tid;
    v[u] = vi < nvec ? load_vec<T, VEC>(p, vi, V)
                     : (std::is_same<T, float>::value
                            ? make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u)
                            : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u));
  }

  // -- thread-local top-2 (values only)
  float t1, t2;
  if constexpr (std::is_same<T, float>::value) {
    t1 = -INFINITY;
    t2 = -INFINITY;
#pragma unroll
    for (int u = 0; u < kConfU; ++u) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float x = elem_of<T>(v[u], e);
        t2 = fmaxf(t2, fminf(t1, x));
        t1 = fmaxf(t1, x);
      }
    }
  } else {
    // two independent packed (max, second) pairs for ILP
    const __nv_bfloat162 ninf = __halves2bfloat162(__ushort_as_bfloat16(0xff80), __ushort_as_bfloat16(0xff80));
    __nv_bfloat162 m1[2] = {ninf, ninf}, m2[2] = {ninf, ninf};
#pragma unroll
    for (int u = 0; u < kConfU; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
        m2[k & 1] = __hmax2(m2[k & 1], __hmin2(m1[k & 1], x));
        m1[k & 1] = __hmax2(m1[k & 1], x);
      }
    }
    m2[0] = __hmax2(__hmax2(m2[0], m2[1]), __hmin2(m1[0], m1[1]));
    m1[0] = __hmax2(m1[0], m1[1]);
    const float a = __bfloat162float(m1[0].x), c = __bfloat162float(m1[0].y);
    t1 = fmaxf(a, c);
    t2 = fmaxf(fminf(a, c), fmaxf(__bfloat162float(m2[0].x), __bfloat162float(m2[0].y)));
  }
  // -- block top-2
  __shared__ float s_t1[kConfThreads / 32], s_t2[kConfThreads / 32], s_l[kConfThreads / 32];
  __shared__ int s_arg[kConfThreads / 32];
  __shared__ float s_M;
  const int lane = tid & 31, warp = tid >> 5;
  const float own_max = t1;  // the thread's own maximum, for the argmax scan
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float o1 = __shfl_xor_sync(0xffffffffu, t1, o);
    const float o2 = __shfl_xor_sync(0xffffffffu, t2, o);
    const float n2 = fmaxf(fminf(t1, o1), fmaxf(t2, o2));
    t1 = fmaxf(t1, o1);
    t2 = n2;
  }
  if (lane == 0) {
    s_t1[warp] = t1;
    s_t2[warp] = t2;
  }
  __syncthreads();
  float M, S2;
  if (tid == 0) {
    M = s_t1[0];
    S2 = s_t2[0];
    for (int w = 1; w < kConfThreads / 32; ++w) {
      const float o1 = s_t1[w], o2 = s_t2[w];
      const float n2 = fmaxf(fminf(M, o1), fmaxf(S2, o2));
      M = fmaxf(M, o1);
      S2 = n2;
    }
    s_M = M;
    s_t2[0] = S2;
  }
  __syncthreads();
  M = s_M;
  S2 = s_t2[0];

  // -- sum of exp(z - M) and lowest index reaching M
  const float negMl = -M * kLog2e;
  float lacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int u = 0; u < kConfU; ++u) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float x = elem_of<T>(v[u], e);
      lacc[e & 3] += ex2_approx(fmaf(x, kLog2e, negMl));
    }
  }
  float l = (lacc[0] + lacc[1]) + (lacc[2] + lacc[3]);
  // Only threads holding M look for its lowest position; the reverse scan
  // leaves the smallest index (u, then e, ascend with the element index).
  int arg = INT_MAX;
  if (own_max == M) {
#pragma unroll
    for (int u = kConfU - 1; u >= 0; --u)
#pragma unroll
      for (int e = E - 1; e >= 0; --e)
        if (elem_of<T>(v[u], e) == M) arg = (vbase + u * kConfThreads + tid) * E + e;
  }
  l = warp_sum(l);
  arg = warp_min_int(arg);
  if (lane == 0) {
    s_l[warp] = l;
    s_arg[warp] = arg;
  }
  __syncthreads();
  if (tid == 0) {
    float lt = 0.f;
    int at = INT_MAX;
    for (int w = 0; w < kConfThreads / 32; ++w) {
      lt += s_l[w];
      at = min(at, s_arg[w]);
    }
    ConfPartial out;
    out.m1 = M;
    out.m2 = S2;
    out.l = lt;
    out.arg = at;
    ws[(int64_t)br * nchunks + chunk] = out;
  }
}

__global__ void conf_merge_kernel(int B, int R_src, int R_max, const int32_t* row_idx,
                                  const int32_t* count,
                                  const int32_t* out_idx, int out_cols, int nchunks,
                                  const ConfPartial* ws, float* conf_out,
                                  int32_t* argmax_out, float* margin_out,
                                  int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t br = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (br >= (int64_t)B * R_max) return;
  const int b = (int)(br / R_max), r = (int)(br - (int64_t)b * R_max);
  int row;
  bool bad;
  const bool ok = row_valid(b, r, R_max, R_src, row_idx, count, &row, &bad);
  if (bad && lane == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
  if (!ok) return;
  int col = r;
  if (out_idx != nullptr) {
    col = __ldca(out_idx + br);
    if (col < 0 || col >= out_cols) {
      if (lane == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
      return;
    }
  }
  ConfPartial acc;
  acc.m1 = -INFINITY;
  acc.m2 = -INFINITY;
  acc.l = 0.f;
  acc.arg = INT_MAX;
  for (int c = lane; c < nchunks; c += 32) {
    const ConfPartial* src = ws + br * nchunks + c;
    ConfPartial w;
    const float4 raw = __ldca(reinterpret_cast<const float4*>(src));
    w.m1 = raw.x;
    w.m2 = raw.y;
    w.l = raw.z;
    w.arg = __float_as_int(raw.w);
    acc = merge(acc, w);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ConfPartial other;
    other.m1 = __shfl_xor_sync(0xffffffffu, acc.m1, o);
    other.m2 = __shfl_xor_sync(0xffffffffu, acc.m2, o);
    other.l = __shfl_xor_sync(0xffffffffu, acc.l, o);
    other.arg = __shfl_xor_sync(0xffffffffu, acc.arg, o);
    acc = merge(acc, other);
  }
  if (lane == 0) {
    const int64_t o = (int64_t)b * out_cols + col;
    conf_out[o] = 1.0f / acc.l;
    argmax_out[o] = acc.arg;
    if (margin_out != nullptr) margin_out[o] = acc.m1 - acc.m2;
  }
}

// ---------------------------------------------------------------------------
// Streaming variant (rows 16-byte aligned, V * sizeof(T) a multiple of 16):
// one persistent CTA per SM.  A producer warp copies 64 KB row chunks with
// cp.async.bulk into a 3-stage shared-memory ring (up to 192 KB of HBM reads
// in flight per SM) and tells the consumers which (row, chunk) each stage
// holds through shared memory.  Each of the 16 consumer warps reduces its own
// 4 KB slice of every staged chunk (64 elements per lane) with warp shuffles
// only, no block barrier, and writes one ConfPartial per slice; the merge
// kernel folds the 16 slices x chunks of a row.  The exponentials run on
// packed f32x2 FMA/add with MUFU ex2 (the MUFU pipe is far from saturated
// here; the limit is latency, hence four consumer warps per scheduler).
// Work items are the valid (row, chunk) pairs in row-major order, dealt
// round-robin to the CTAs (neighbouring chunks stream at the same time).
constexpr int kStreamMaxB = 64;  // batch rows whose counts are staged in shared memory
constexpr int kStreamWarps = 16;                         // consumer warps
constexpr int kStreamThreads = (kStreamWarps + 1) * 32;
constexpr int kStreamStages = 3;
constexpr uint32_t kStreamChunkBytes = 65536;
constexpr uint32_t kStreamSliceBytes = kStreamChunkBytes / kStreamWarps;  // 4 KB per warp
constexpr int kStreamVPL = kStreamSliceBytes / 16 / 32;                   // 16-byte vectors per lane
constexpr uint32_t kStreamSmem = kStreamStages * kStreamChunkBytes + 256 + 1024;

__host__ __device__ inline int stream_nchunks(int V, int elem_bytes) {
  const int64_t bytes = (int64_t)V * elem_bytes;
  const int n = (int)((bytes + kStreamChunkBytes - 1) / kStreamChunkBytes);
  return n < 1 ? 1 : n;
}

__device__ __forceinline__ uint4 ld_shared16(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}

// Whether any element of the 16-byte vector equals m (m is not NaN).
template <typename T>
__device__ __forceinline__ bool vec_contains(const uint4& v, float m) {
  if constexpr (std::is_same<T, float>::value) {
    return __uint_as_float(v.x) == m || __uint_as_float(v.y) == m ||
           __uint_as_float(v.z) == m || __uint_as_float(v.w) == m;
  } else {
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.x),
                                     *reinterpret_cast<const __nv_bfloat162*>(&v.y));
    const __nv_bfloat162 c = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.z),
                                     *reinterpret_cast<const __nv_bfloat162*>(&v.w));
    const __nv_bfloat162 mx = __hmax2(a, c);
    // m is the maximum of a set that contains these elements, so equality
    // with the vector's maximum is the test
    return fmaxf(__bfloat162float(mx.x), __bfloat162float(mx.y)) == m;
  }
}

// Lane top-1 and top-2 over the lane's vectors (packed bf16x2 pairs of
// (max, second) in four independent chains for bf16).
template <typename T>
__device__ __forceinline__ void lane_top2(const uint4 (&x)[kStreamVPL], float* m1, float* m2) {
  constexpr int E = vec_elems<T>();
  if constexpr (std::is_same<T, float>::value) {
    float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
    for (int u = 0; u < kStreamVPL; ++u)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float z = elem_of<T>(x[u], e);
        t2 = fmaxf(t2, fminf(t1, z));
        t1 = fmaxf(t1, z);
      }
    *m1 = t1;
    *m2 = t2;
  } else {
    const __nv_bfloat162 ninf =
        __halves2bfloat162(__ushort_as_bfloat16(0xff80), __ushort_as_bfloat16(0xff80));
    __nv_bfloat162 a1[4] = {ninf, ninf, ninf, ninf}, a2[4] = {ninf, ninf, ninf, ninf};
#pragma unroll
    for (int u = 0; u < kStreamVPL; ++u) {
      const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 z = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
        a2[k] = __hmax2(a2[k], __hmin2(a1[k], z));
        a1[k] = __hmax2(a1[k], z);
      }
    }
#pragma unroll
    for (int k = 1; k < 4; ++k) {
      a2[0] = __hmax2(__hmax2(a2[0], a2[k]), __hmin2(a1[0], a1[k]));
      a1[0] = __hmax2(a1[0], a1[k]);
    }
    const float p = __bfloat162float(a1[0].x), q = __bfloat162float(a1[0].y);
    *m1 = fmaxf(p, q);
    *m2 = fmaxf(fminf(p, q), fmaxf(__bfloat162float(a2[0].x), __bfloat162float(a2[0].y)));
  }
}

// Lane sum of 2^(z log2 e + nm) over the lane's vectors (nm = -M log2 e).
template <typename T>
__device__ __forceinline__ float lane_sumexp(const uint4 (&x)[kStreamVPL], float nm) {
  if constexpr (std::is_same<T, float>::value) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < kStreamVPL; ++u) {
      acc[0] += ex2_approx(fmaf(__uint_as_float(x[u].x), kLog2e, nm));
      acc[1] += ex2_approx(fmaf(__uint_as_float(x[u].y), kLog2e, nm));
      acc[2] += ex2_approx(fmaf(__uint_as_float(x[u].z), kLog2e, nm));
      acc[3] += ex2_approx(fmaf(__uint_as_float(x[u].w), kLog2e, nm));
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
  } else {
    const float2 l2e = make_float2(kLog2e, kLog2e);
    const float2 n2 = make_float2(nm, nm);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int u = 0; u < kStreamVPL; ++u) {
      const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 a = __ffma2_rn(make_float2(bf16_lo(w[k]), bf16_hi(w[k])), l2e, n2);
        const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
        if (k & 1)
          acc1 = __fadd2_rn(acc1, e);
        else
          acc0 = __fadd2_rn(acc0, e);
      }
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
  }
}

template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 1)
conf_stream_kernel(const T* logits, int R_src, int V, int64_t rs, int64_t bs,
                   int B, int R_max, const int32_t* row_idx,
                   const int32_t* count, int nchunks,
                   ConfPartial* ws, int32_t* dev_status, long long wait_limit) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  using namespace sm100;
  constexpr int E = vec_elems<T>();
  constexpr int CE = kStreamChunkBytes / sizeof(T);  // elements per chunk
  constexpr int SE = kStreamSliceBytes / sizeof(T);  // elements per warp slice
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(gbase + kStreamStages * kStreamChunkBytes);
  uint64_t* empty = full + kStreamStages;
  int* abort_flag = reinterpret_cast<int*>(empty + kStreamStages);
  // (batch row * R_max + row, chunk) of each staged chunk; br < 0 ends the stream
  int2* stage_info = reinterpret_cast<int2*>(abort_flag + 2);

  __shared__ int s_cnt[kStreamMaxB];  // clamped counts of the first batch rows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStreamStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kStreamWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  for (int b = tid; b < B && b < kStreamMaxB; b += blockDim.x) {
    const int n = count ? __ldca(count + b) : R_max;
    s_cnt[b] = n < 0 ? 0 : (n > R_max ? R_max : n);
  }
  __syncthreads();
  volatile int* abort = abort_flag;

  if (warp == kStreamWarps) {
    // ------------------------------------------------------------ producer
    // The producer alone reads counts and row indices; the consumers learn
    // which row and chunk each stage holds from stage_info.
    if (lane == 0) {
      // Valid items only, in row-major order ((b, r < count[b], chunk)),
      // dealt round-robin: at any time the CTAs stream neighbouring chunks.
      auto cnt = [&](int b) {
        if (b < kStreamMaxB) return s_cnt[b];
        int n = count ? __ldca(count + b) : R_max;
        return n < 0 ? 0 : (n > R_max ? R_max : n);  // out of range: reported by the merge kernel
      };
      int64_t rows = 0;
      for (int b = 0; b < B; ++b) rows += cnt(b);
      const int64_t total = rows * nchunks;
      int j = 0, b = 0;
      int64_t row_base = 0;  // valid rows before batch row b
      bool ok = true;
      for (int64_t v = blockIdx.x; v < total; v += gridDim.x) {
        const int64_t vr = v / nchunks;
        const int c = (int)(v - vr * nchunks);
        while (vr >= row_base + cnt(b)) row_base += cnt(b++);
        const int r = (int)(vr - row_base);
        const int br = b * R_max + r;
        const int row = row_idx ? __ldca(row_idx + br) : r;
        if (row < 0 || row >= R_src) continue;  // the merge kernel reports it
        const int stage = j % kStreamStages;
        if (j >= kStreamStages &&
            !mbar_wait(&empty[stage], ((j / kStreamStages) - 1) & 1, abort, wait_limit)) {
          ok = false;
          break;
        }
        stage_info[stage] = make_int2(br, c);
        const int e0 = c * CE;
        const uint32_t bytes = (uint32_t)min(CE, V - e0) * (uint32_t)sizeof(T);
        mbar_expect_tx(&full[stage], bytes);
        bulk_load(gbase + stage * kStreamChunkBytes,
                  logits + (int64_t)b * bs + (int64_t)row * rs + e0, bytes, &full[stage]);
        ++j;
      }
      bool sentinel = false;
      if (ok) {  // end-of-stream stage: a plain arrival with br = -1
        const int stage = j % kStreamStages;
        if (j < kStreamStages || mbar_wait(&empty[stage], ((j / kStreamStages) - 1) & 1, abort, wait_limit)) {
          stage_info[stage] = make_int2(-1, 0);
          mbar_arrive(&full[stage]);
          sentinel = true;
        }
      }
      // Never leave with copies in flight into shared memory: wait for the
      // data stages that may still be loading.  After the sentinel, the use
      // j - kStreamStages of its stage is known to be consumed, and that
      // stage's barrier has moved one phase further, so it is left out.
      int none = 0;
      int k0 = j - kStreamStages + (sentinel ? 1 : 0);
      for (int k = k0 < 0 ? 0 : k0; k < j; ++k)
        mbar_wait(&full[k % kStreamStages], (k / kStreamStages) & 1, &none);
      if (none) report(dev_status, DLLM_ERR_TIMEOUT);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const uint32_t sent = std::is_same<T, float>::value ? 0xff800000u : 0xff80ff80u;
  for (int j = 0;; ++j) {
    const int stage = j % kStreamStages;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], (j / kStreamStages) & 1, abort, wait_limit))) break;
    const int2 info = stage_info[stage];
    if (info.x < 0) break;
    const int br = info.x, c = info.y;
    const int s0 = c * CE + warp * SE;  // first element of this warp's slice
    const int nvec = max(0, min(SE, V - s0)) / E;
    const uint32_t sbase = base + stage * kStreamChunkBytes + warp * kStreamSliceBytes;
    uint4 x[kStreamVPL];
    if (nvec == kStreamVPL * 32) {  // full slice: no bounds test per vector
#pragma unroll
      for (int u = 0; u < kStreamVPL; ++u) x[u] = ld_shared16(sbase + (u * 32 + lane) * 16);
    } else {
#pragma unroll
      for (int u = 0; u < kStreamVPL; ++u) {
        const int vi = u * 32 + lane;
        x[u] = vi < nvec ? ld_shared16(sbase + vi * 16) : make_uint4(sent, sent, sent, sent);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);  // this warp's slice is in registers
    // Slice top-2 first (lane chains, then a shuffle tree), then the sum of
    // exp(z - M) relative to the slice maximum M directly, so no partial
    // sums need rescaling; lanes holding M find its lowest position.
    float own_max, own_2;
    lane_top2<T>(x, &own_max, &own_2);
    float t1 = own_max, t2 = own_2;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float o1 = __shfl_xor_sync(0xffffffffu, t1, o);
      const float o2 = __shfl_xor_sync(0xffffffffu, t2, o);
      t2 = fmaxf(fminf(t1, o1), fmaxf(t2, o2));
      t1 = fmaxf(t1, o1);
    }
    const float lsum = t1 == -INFINITY ? 0.f : warp_sum(lane_sumexp<T>(x, -t1 * kLog2e));
    int arg = INT_MAX;
    if (own_max == t1 && own_max != -INFINITY) {
      // usually one lane: the first vector containing the maximum, then the
      // first element in it (indices ascend with u, then e)
#pragma unroll
      for (int u = 0; u < kStreamVPL; ++u) {
        if (arg == INT_MAX && vec_contains<T>(x[u], t1)) {
#pragma unroll
          for (int e = E - 1; e >= 0; --e)
            if (elem_of<T>(x[u], e) == t1) arg = s0 + (u * 32 + lane) * E + e;
        }
      }
    }
    arg = __reduce_min_sync(0xffffffffu, arg);
    if (lane == 0) {
      ConfPartial out;
      out.m1 = t1;
      out.m2 = t2;
      out.l = lsum;
      out.arg = arg;
      ws[((int64_t)br * nchunks + c) * kStreamWarps + warp] = out;
    }
  }
  if (lane == 0 && *abort) report(dev_status, DLLM_ERR_TIMEOUT);
}

template <typename T>
int conf_nchunks(int V) {
  const int n = (V + conf_chunk_elems<T>() - 1) / conf_chunk_elems<T>();
  return n < 1 ? 1 : n;
}

template <typename T>
cudaError_t launch_typed(const T* logits, int B, int R_src, int V, int64_t rs, int64_t bs,
                         int R_max, const int32_t* row_idx, const int32_t* count,
                         const int32_t* out_idx, int out_cols, float* conf_out,
                         int32_t* argmax_out, float* margin_out, void* ws, int32_t* dev_status,
                         cudaStream_t stream) {
  constexpr int E = vec_elems<T>();
  const int nchunks = conf_nchunks<T>(V);
  const bool vec = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && (rs % E == 0) &&
                   (bs % E == 0);
  ConfPartial* part = static_cast<ConfPartial*>(ws);
  int parts = nchunks;  // partials per row handed to the merge
  const bool stream_ok = vec && ((int64_t)V * (int64_t)sizeof(T)) % 16 == 0 &&
                         (int64_t)B * R_max * stream_nchunks(V, (int)sizeof(T)) < INT32_MAX;
  if (stream_ok) {
    const cudaError_t ea =
        ensure_smem_limit(reinterpret_cast<const void*>(conf_stream_kernel<T>), (int)kStreamSmem);
    if (ea != cudaSuccess) return ea;
    const int snc = stream_nchunks(V, (int)sizeof(T));
    launch_pdl(conf_stream_kernel<T>, num_sms(), kStreamThreads, kStreamSmem, stream,
        logits, R_src, V, rs, bs, B, R_max, row_idx, count, snc, part, dev_status,
        wait_limit());
    parts = snc * kStreamWarps;
  } else {
    dim3 grid(B * R_max, nchunks);
    if (vec)
      launch_pdl(conf_partial_kernel<T, true>, grid, kConfThreads, 0, stream,
          logits, R_src, V, rs, bs, R_max, row_idx, count, nchunks, part);
    else
      launch_pdl(conf_partial_kernel<T, false>, grid, kConfThreads, 0, stream,
          logits, R_src, V, rs, bs, R_max, row_idx, count, nchunks, part);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t rows = (int64_t)B * R_max;
  const int warps = 8;
  launch_pdl(conf_merge_kernel, (unsigned)((rows + warps - 1) / warps), warps * 32, 0, stream,
      B, R_src, R_max, row_idx, count, out_idx, out_cols, parts, part, conf_out, argmax_out,
      margin_out, dev_status);
  return cudaGetLastError();
}

}  // namespace

size_t confidence_workspace_bytes(int B, int R_max, int V, int dtype) {
  // partials per row: one per 32 KB chunk (chunked kernel) or one per 4 KB
  // slice (kStreamSliceBytes, streaming kernel); size for the larger
  const int eb = dtype == DLLM_BF16 ? 2 : 4;
  const int a = dtype == DLLM_BF16 ? conf_nchunks<__nv_bfloat16>(V) : conf_nchunks<float>(V);
  const int s = stream_nchunks(V, eb) * kStreamWarps;
  return (size_t)B * (size_t)R_max * (size_t)(a > s ? a : s) * sizeof(ConfPartial);
}

cudaError_t launch_confidence(const void* logits, int dtype, int B, int R_src, int V,
                              int64_t row_stride, int64_t batch_stride, int R_max,
                              const int32_t* row_idx, const int32_t* count,
                              const int32_t* out_idx, int out_cols, float* conf_out,
                              int32_t* argmax_out, float* margin_out, void* ws,
                              int32_t* dev_status, cudaStream_t stream) {
  if (dtype == DLLM_BF16)
    return launch_typed(static_cast<const __nv_bfloat16*>(logits), B, R_src, V, row_stride,
                        batch_stride, R_max, row_idx, count, out_idx, out_cols, conf_out,
                        argmax_out, margin_out, ws, dev_status, stream);
  return launch_typed(static_cast<const float*>(logits), B, R_src, V, row_stride, batch_stride,
                      R_max, row_idx, count, out_idx, out_cols, conf_out, argmax_out,
                      margin_out, ws, dev_status, stream);
}

}  // namespace dllm
