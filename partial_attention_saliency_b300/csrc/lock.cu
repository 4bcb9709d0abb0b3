// Lock criterion between consecutive steps, and the adaptive prefix threshold.
//
// SureLock ("Stopping Computation for Converged Tokens in Masked Diffusion-LM
// Decoding"), technical summary section 2, locking criterion 1: a position
// locks when the local divergence D = KL(p_t || p_{t-1}) of its predictive
// distribution between two steps falls below eps; criterion 2 (optional):
// its uncertainty 1 - max p_t must lie below a percentile.  LSP ("Beyond
// Scattered Acceptance ..."), technical summary section 2, step 2: the
// threshold of the stable prefix is chosen so that the committed block
// covers a fraction [lo, hi] of the active length.
//
// lock_partial_persistent_kernel / lock_partial_kernel
//                      one CTA per (row, chunk of 256 kLockU 16-byte vectors
//                      of each of the two logit rows) -- persistent CTAs
//                      over the valid items up to 64 batch rows, a grid of
//                      all row slots above: every thread sums
//                      exp(z - mz), exp(z - mz)(z - y) and exp(y - my) over
//                      its own elements relative to its own maxima, then
//                      rescales them to the block maxima (one exchange) and
//                      the block adds them up; HBM bound, 2 V sizeof(T) per
//                      row.
// lock_merge_kernel    one warp per row folds the chunks in a fixed order and
//                      evaluates KL = A / lz - (Mz + ln lz) + (My + ln ly) in
//                      double; the uncertainty is 1 - 1 / lz.
//                      With the confidence (a second instantiation of the
//                      partial and merge kernels), the same pass also keeps
//                      the top two current logits and the lowest index of the
//                      top one, and the merge writes the confidence 1 / lz,
//                      that index and the margin: dllm_confidence's outputs
//                      without a second read of the current row.
// lock_gate_kernel     one CTA per batch row: radix select of the k-th
//                      smallest uncertainty among the active rows (the
//                      percentile gate), then the lock flags (only ever set).
// adaptive_prefix_kernel one CTA per batch row: block-wide prefix-minimum scan
//                      of the active suffix, tau at ceil(lo A), the run of
//                      prefix minima >= tau capped at floor(hi A).
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kLockThreads = 256;
// Tuned on bf16 rows of 126464 logits: 4 16-byte vectors per thread and
// input with at least 4 CTAs per SM (64 registers, a 56-byte spill) ran at
// 333 us for 2867 rows, against 370 us at 3 CTAs per SM, 388 us with 2
// vectors and 518 us with 8.  Taking a quarter to a half of the previous
// row's exponentials from an FMA-pipe polynomial instead of the SFU was
// slower (457 to 476 us): the SFU is not the limit here.
#ifndef DLLM_LOCK_U
#define DLLM_LOCK_U 4
#endif
#ifndef DLLM_LOCK_MINB
#define DLLM_LOCK_MINB 4
#endif
constexpr int kLockU = DLLM_LOCK_U;  // 16-byte vectors per thread per chunk and input
constexpr int kGateThreads = 1024;
constexpr int kGateMaxRows = 16384;  // uncertainty keys held in shared memory (64 KB)
constexpr int kLockMaxB = 64;        // batch rows the persistent partial kernel stages

struct LockPartial {
  float mz, lz, a, my, ly;
  float m2z;   // with the confidence: second largest current logit (mz on a tie)
  int argz;    // with the confidence: lowest index of mz
  float pad;   // 32 bytes
};

// Shared scratch of one CTA's reduction.
struct LockRed {
  float max[2][kLockThreads / 32];
  float sum[3][kLockThreads / 32];
  float m2[kLockThreads / 32];  // with the confidence
  int arg[kLockThreads / 32];
};

// (top, second, lowest index of top) of two sets, the second counting ties.
__device__ __forceinline__ void top2_merge(float& m1, float& m2, int& arg, float o1, float o2,
                                           int oa) {
  if (o1 > m1) {
    m2 = fmaxf(o2, m1);
    m1 = o1;
    arg = oa;
  } else if (o1 < m1) {
    m2 = fmaxf(m2, o1);
  } else {
    m2 = m1;
    arg = min(arg, oa);
  }
}

template <typename T> __host__ __device__ constexpr int lvec() { return 16 / (int)sizeof(T); }
template <typename T> __host__ __device__ constexpr int lock_chunk_elems() {
  return kLockThreads * kLockU * lvec<T>();
}

template <typename T>
__device__ __forceinline__ float lelem(const uint4& v, int e) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (std::is_same<T, float>::value) {
    return __uint_as_float(w[e]);
  } else {
    return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
  }
}

template <typename T, bool VEC>
__device__ __forceinline__ uint4 lload(const T* row, int vi, int V) {
  constexpr int E = lvec<T>();
  if (VEC && (vi + 1) * E <= V) return ld_stream16(row + (int64_t)vi * E);
  uint32_t w[4];
  if constexpr (std::is_same<T, float>::value) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = vi * E + k;
      w[k] = i < V ? __float_as_uint(row[i]) : 0xff800000u;
    }
  } else {
    const uint16_t* hh = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i0 = vi * E + 2 * k, i1 = i0 + 1;
      const uint32_t lo = i0 < V ? hh[i0] : 0xff80u;
      const uint32_t hi = i1 < V ? hh[i1] : 0xff80u;
      w[k] = lo | (hi << 16);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ bool lock_row(int b, int r, int R_max, int R_src,
                                         const int32_t* row_idx, const int32_t* count, int* row,
                                         bool* bad) {
  int n = count ? __ldca(count + b) : R_max;
  *bad = false;
  if (n < 0 || n > R_max) {
    *bad = true;
    n = n < 0 ? 0 : R_max;
  }
  if (r >= n) return false;
  const int rr = row_idx ? __ldca(row_idx + (int64_t)b * R_max + r) : r;
  if (rr < 0 || rr >= R_src) {
    *bad = true;
    return false;
  }
  *row = rr;
  return true;
}

// This thread's vectors of one (row, chunk): zrow / yrow point at the two
// logit rows; -inf past the row end.
template <typename T, bool VEC>
__device__ __forceinline__ void lock_load(const T* zrow, const T* yrow, int V, int chunk,
                                          uint4 (&vz)[kLockU], uint4 (&vy)[kLockU]) {
  constexpr int E = lvec<T>();
  const int vbase = chunk * (kLockThreads * kLockU);
  const int nvec = (V + E - 1) / E;
  const uint32_t sent = std::is_same<T, float>::value ? 0xff800000u : 0xff80ff80u;
#pragma unroll
  for (int u = 0; u < kLockU; ++u) {
    const int vi = vbase + u * kLockThreads + threadIdx.x;
    vz[u] = vi < nvec ? lload<T, VEC>(zrow, vi, V) : make_uint4(sent, sent, sent, sent);
    vy[u] = vi < nvec ? lload<T, VEC>(yrow, vi, V) : make_uint4(sent, sent, sent, sent);
  }
}

// The partial of one (row, chunk) from the CTA's loaded vectors; thread 0
// writes it to *out_slot.  CONF: also the top two current logits and the
// lowest index of the top one.
template <typename T, bool CONF>
__device__ __forceinline__ void lock_reduce(const uint4 (&vz)[kLockU], const uint4 (&vy)[kLockU],
                                            int chunk, LockPartial* out_slot, LockRed& red) {
  constexpr int E = lvec<T>();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // 1. this thread's maxima and its sums relative to them: no block-wide
  //    step before the exponentials
  float mz = -INFINITY, my = -INFINITY, m2z = -INFINITY;
  int argz = INT_MAX;
  if constexpr (CONF) {
#pragma unroll
    for (int u = 0; u < kLockU; ++u)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float x = lelem<T>(vz[u], e);
        m2z = fmaxf(m2z, fminf(mz, x));
        mz = fmaxf(mz, x);
      }
#pragma unroll
    for (int u = 0; u < kLockU; ++u)
#pragma unroll
      for (int e = 0; e < E; e += 2) my = fmax3(my, lelem<T>(vy[u], e), lelem<T>(vy[u], e + 1));
    if (mz != -INFINITY) {
      // elements ascend with u, then e: the first match is the lowest index
      const int vbase = chunk * (kLockThreads * kLockU);
#pragma unroll
      for (int u = kLockU - 1; u >= 0; --u)
#pragma unroll
        for (int e = E - 1; e >= 0; --e)
          if (lelem<T>(vz[u], e) == mz)
            argz = (vbase + u * kLockThreads + (int)threadIdx.x) * E + e;
    }
  } else {
#pragma unroll
    for (int u = 0; u < kLockU; ++u)
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        mz = fmax3(mz, lelem<T>(vz[u], e), lelem<T>(vz[u], e + 1));
        my = fmax3(my, lelem<T>(vy[u], e), lelem<T>(vy[u], e + 1));
      }
  }
  float lz = 0.f, a = 0.f, ly = 0.f;
  if (mz != -INFINITY) {
    const float nz = -mz * kLog2e, ny = -my * kLog2e;
#pragma unroll
    for (int u = 0; u < kLockU; ++u)
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float z0 = lelem<T>(vz[u], e), z1 = lelem<T>(vz[u], e + 1);
        const float y0 = lelem<T>(vy[u], e), y1 = lelem<T>(vy[u], e + 1);
        const float p0 = ex2_approx(fmaf(z0, kLog2e, nz));
        const float p1 = ex2_approx(fmaf(z1, kLog2e, nz));
        const float q0 = ex2_approx(fmaf(y0, kLog2e, ny));
        const float q1 = ex2_approx(fmaf(y1, kLog2e, ny));
        // padding past the row end holds -inf in both rows: no contribution
        if (z0 != -INFINITY) {
          lz += p0;
          a = fmaf(p0, z0 - y0, a);
          ly += q0;
        }
        if (z1 != -INFINITY) {
          lz += p1;
          a = fmaf(p1, z1 - y1, a);
          ly += q1;
        }
      }
  }
  // 2. block maxima (one exchange), each thread rescales its own sums
  float wz = mz;
  if constexpr (CONF) {
    float w2 = m2z;
    int wa = argz;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float o1 = __shfl_xor_sync(0xffffffffu, wz, off);
      const float o2 = __shfl_xor_sync(0xffffffffu, w2, off);
      const int oa = __shfl_xor_sync(0xffffffffu, wa, off);
      top2_merge(wz, w2, wa, o1, o2, oa);
    }
    if (lane == 0) {
      red.m2[warp] = w2;
      red.arg[warp] = wa;
    }
  } else {
    wz = warp_max(mz);
  }
  const float wy = warp_max(my);
  if (lane == 0) {
    red.max[0][warp] = wz;
    red.max[1][warp] = wy;
  }
  __syncthreads();
  float Mz = red.max[0][0], My = red.max[1][0];
#pragma unroll
  for (int w = 1; w < kLockThreads / 32; ++w) {
    Mz = fmaxf(Mz, red.max[0][w]);
    My = fmaxf(My, red.max[1][w]);
  }
  // the block's second logit and index, read before the next barrier (after
  // it, a warp may already be writing the next item's maxima)
  float bm2 = -INFINITY;
  int barg = INT_MAX;
  if (CONF && threadIdx.x == 0) {
    float m1 = red.max[0][0];
    bm2 = red.m2[0];
    barg = red.arg[0];
    for (int w = 1; w < kLockThreads / 32; ++w)  // fixed order
      top2_merge(m1, bm2, barg, red.max[0][w], red.m2[w], red.arg[w]);
  }
  const float cz = mz == -INFINITY ? 0.f : ex2_approx((mz - Mz) * kLog2e);
  const float cy = my == -INFINITY ? 0.f : ex2_approx((my - My) * kLog2e);
  lz = warp_sum(lz * cz);
  a = warp_sum(a * cz);
  ly = warp_sum(ly * cy);
  if (lane == 0) {
    red.sum[0][warp] = lz;
    red.sum[1][warp] = a;
    red.sum[2][warp] = ly;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    LockPartial out;
    out.mz = Mz;
    out.my = My;
    out.lz = out.a = out.ly = 0.f;
    for (int w = 0; w < kLockThreads / 32; ++w) {  // fixed order
      out.lz += red.sum[0][w];
      out.a += red.sum[1][w];
      out.ly += red.sum[2][w];
    }
    out.m2z = bm2;
    out.argz = barg;
    out.pad = 0.f;
    *out_slot = out;
  }
}

// One CTA per (row slot, chunk): slots past their batch row's count exit at
// once.  For batch counts beyond kLockMaxB.
template <typename T, bool VEC, bool CONF>
__global__ void __launch_bounds__(kLockThreads, DLLM_LOCK_MINB)
lock_partial_kernel(const T* zs, const T* ys, int R_src, int V, int64_t rs, int64_t bs, int R_max,
                    const int32_t* row_idx, const int32_t* count, int nchunks, LockPartial* ws) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  __shared__ LockRed red;
  const int br = blockIdx.x, chunk = blockIdx.y;
  const int b = br / R_max, r = br - b * R_max;
  int row;
  bool bad;
  if (!lock_row(b, r, R_max, R_src, row_idx, count, &row, &bad)) return;
  uint4 vz[kLockU], vy[kLockU];
  lock_load<T, VEC>(zs + (int64_t)b * bs + (int64_t)row * rs,
                    ys + (int64_t)b * bs + (int64_t)row * rs, V, chunk, vz, vy);
  lock_reduce<T, CONF>(vz, vy, chunk, ws + (int64_t)br * nchunks + chunk, red);
}

// Persistent: the CTAs take the valid (row, chunk) items, row-major, dealt
// round-robin from the counts (staged once per CTA), so no CTA is spent on
// the row slots past the counts (a grid over every row slot of a 1024-slot
// window with 124 active rows per batch row took 108 us, this kernel 83 us;
// 77 us and 81 us with 128 slots).  Rows whose index is out of range are
// skipped (the merge kernel reports them).
template <typename T, bool VEC, bool CONF>
__global__ void __launch_bounds__(kLockThreads, DLLM_LOCK_MINB)
lock_partial_persistent_kernel(const T* zs, const T* ys, int R_src, int V, int64_t rs,
                               int64_t bs, int B, int R_max, const int32_t* row_idx,
                               const int32_t* count, int nchunks, LockPartial* ws) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  __shared__ LockRed red;
  __shared__ int s_pre[kLockMaxB + 1];  // valid rows before each batch row
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      int n = count ? __ldca(count + b) : R_max;
      n = n < 0 ? 0 : (n > R_max ? R_max : n);  // out of range: reported by the merge kernel
      s_pre[b] = acc;
      acc += n;
    }
    s_pre[B] = acc;
  }
  __syncthreads();
  const int64_t total = (int64_t)s_pre[B] * nchunks;
  int b = 0;  // items ascend, so the batch row only grows
  // the next valid item at or after v: its rows and output slot
  auto next = [&](int64_t v, int64_t* at, const T** zr, const T** yr, int* chunk,
                  LockPartial** slot) {
    for (; v < total; v += gridDim.x) {
      const int vr = (int)(v / nchunks);
      *chunk = (int)(v - (int64_t)vr * nchunks);
      while (vr >= s_pre[b + 1]) ++b;
      const int r = vr - s_pre[b];
      const int64_t br = (int64_t)b * R_max + r;
      const int row = row_idx ? __ldca(row_idx + br) : r;
      if (row < 0 || row >= R_src) continue;  // CTA-uniform
      *zr = zs + (int64_t)b * bs + (int64_t)row * rs;
      *yr = ys + (int64_t)b * bs + (int64_t)row * rs;
      *slot = ws + br * nchunks + *chunk;
      *at = v;
      return true;
    }
    *at = total;
    return false;
  };
  int64_t v = blockIdx.x;
  const T *zr, *yr;
  int chunk;
  LockPartial* slot;
  uint4 za[kLockU], ya[kLockU];
  while (next(v, &v, &zr, &yr, &chunk, &slot)) {
    lock_load<T, VEC>(zr, yr, V, chunk, za, ya);
    lock_reduce<T, CONF>(za, ya, chunk, slot, red);
    v += gridDim.x;
  }
}

struct LockAcc {
  float mz, lz, a, my, ly, m2z;
  int argz;
};

template <bool CONF>
__device__ __forceinline__ LockAcc lock_fold(const LockAcc& p, const LockAcc& q) {
  LockAcc r;
  r.m2z = -INFINITY;
  r.argz = INT_MAX;
  if constexpr (CONF) {
    float m1 = p.mz;
    r.m2z = p.m2z;
    r.argz = p.argz;
    top2_merge(m1, r.m2z, r.argz, q.mz, q.m2z, q.argz);
  }
  r.mz = fmaxf(p.mz, q.mz);
  r.my = fmaxf(p.my, q.my);
  const float cp = p.mz == -INFINITY ? 0.f : ex2_approx((p.mz - r.mz) * kLog2e);
  const float cq = q.mz == -INFINITY ? 0.f : ex2_approx((q.mz - r.mz) * kLog2e);
  const float dp = p.my == -INFINITY ? 0.f : ex2_approx((p.my - r.my) * kLog2e);
  const float dq = q.my == -INFINITY ? 0.f : ex2_approx((q.my - r.my) * kLog2e);
  r.lz = p.lz * cp + q.lz * cq;
  r.a = p.a * cp + q.a * cq;
  r.ly = p.ly * dp + q.ly * dq;
  return r;
}

template <bool CONF>
__global__ void lock_merge_kernel(int B, int R_src, int R_max, const int32_t* row_idx,
                                  const int32_t* count, const int32_t* out_idx, int out_cols,
                                  int nchunks, const LockPartial* ws, float* kl_out,
                                  float* unc_out, float* conf_out, int32_t* argmax_out,
                                  float* margin_out, int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t br = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (br >= (int64_t)B * R_max) return;
  const int b = (int)(br / R_max), r = (int)(br - (int64_t)b * R_max);
  int row;
  bool bad;
  const bool ok = lock_row(b, r, R_max, R_src, row_idx, count, &row, &bad);
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
  LockAcc acc{-INFINITY, 0.f, 0.f, -INFINITY, 0.f, -INFINITY, INT_MAX};
  for (int c = lane; c < nchunks; c += 32) {
    const float4* src = reinterpret_cast<const float4*>(ws + br * nchunks + c);
    const float4 p0 = __ldca(src), p1 = __ldca(src + 1);
    acc = lock_fold<CONF>(acc, LockAcc{p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, __float_as_int(p1.z)});
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    LockAcc o;
    o.mz = __shfl_xor_sync(0xffffffffu, acc.mz, off);
    o.lz = __shfl_xor_sync(0xffffffffu, acc.lz, off);
    o.a = __shfl_xor_sync(0xffffffffu, acc.a, off);
    o.my = __shfl_xor_sync(0xffffffffu, acc.my, off);
    o.ly = __shfl_xor_sync(0xffffffffu, acc.ly, off);
    o.m2z = -INFINITY;
    o.argz = INT_MAX;
    if constexpr (CONF) {
      o.m2z = __shfl_xor_sync(0xffffffffu, acc.m2z, off);
      o.argz = __shfl_xor_sync(0xffffffffu, acc.argz, off);
    }
    acc = lock_fold<CONF>(acc, o);
  }
  if (lane == 0) {
    const double lse_z = (double)acc.mz + log((double)acc.lz);
    const double lse_y = (double)acc.my + log((double)acc.ly);
    const double kl = (double)acc.a / (double)acc.lz - lse_z + lse_y;
    const int64_t o = (int64_t)b * out_cols + col;
    kl_out[o] = (float)kl;
    // lz >= 1 up to rounding (the largest term is exp(0)): clamp at 0
    unc_out[o] = fmaxf(1.0f - 1.0f / acc.lz, 0.0f);
    if constexpr (CONF) {
      conf_out[o] = 1.0f / acc.lz;
      argmax_out[o] = acc.argz;
      if (margin_out != nullptr) margin_out[o] = acc.mz - acc.m2z;
    }
  }
}

// Order-preserving unsigned key of a float (NaN sorts last), and its inverse.
__device__ __forceinline__ uint32_t ukey(float u) {
  if (isnan(u)) return 0xffffffffu;
  const uint32_t x = __float_as_uint(u);
  return (x & 0x80000000u) ? ~x : (x | 0x80000000u);
}
__device__ __forceinline__ float ukey_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__global__ void __launch_bounds__(kGateThreads)
lock_gate_kernel(int R_max, const int32_t* count, const int32_t* out_idx, int out_cols,
                 const float* kl, const float* unc, float eps, float gate_q, uint8_t* locked,
                 int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  extern __shared__ uint32_t keys[];  // [R_max] uncertainty keys of the active rows
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_k;
  const int b = blockIdx.x;
  int n = count ? __ldca(count + b) : R_max;
  n = n < 0 ? 0 : (n > R_max ? R_max : n);
  auto col_of = [&](int r) { return out_idx ? __ldca(out_idx + (int64_t)b * R_max + r) : r; };
  const bool gate = gate_q > 0.f && gate_q < 1.f;
  float t = INFINITY;
  if (gate && n > 0) {
    for (int r = threadIdx.x; r < n; r += blockDim.x) {
      const int c = col_of(r);
      keys[r] = (c >= 0 && c < out_cols) ? ukey(__ldca(unc + (int64_t)b * out_cols + c))
                                         : 0xffffffffu;
    }
    if (threadIdx.x == 0) {
      s_prefix = 0;
      // k = max(1, ceil(q n)), the product of the float32 q and n taken exactly in double
      int k = (int)ceil((double)gate_q * (double)n);
      s_k = (uint32_t)(k < 1 ? 1 : (k > n ? n : k));
    }
    uint32_t mask = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      for (int r = threadIdx.x; r < n; r += blockDim.x) {
        const uint32_t key = keys[r];
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        uint32_t k = s_k, cum = 0;
        int d = 0;
        for (; d < 256; ++d) {
          if (cum + hist[d] >= k) break;
          cum += hist[d];
        }
        s_k = k - cum;
        s_prefix = prefix | ((uint32_t)d << shift);
      }
      mask |= 255u << shift;
      __syncthreads();
    }
    const uint32_t tk = s_prefix;
    t = tk == 0xffffffffu ? INFINITY : ukey_value(tk);
  }
  if (locked == nullptr) return;
  const float e32 = eps;
  for (int r = threadIdx.x; r < n; r += blockDim.x) {
    const int c = col_of(r);
    if (c < 0 || c >= out_cols) continue;  // reported by the merge kernel
    const int64_t o = (int64_t)b * out_cols + c;
    const float d = __ldca(kl + o), u = __ldca(unc + o);
    if (d < e32 && (!gate || u <= t)) locked[o] = 1;
  }
}

constexpr int kPrefixScanThreads = 1024;

__global__ void __launch_bounds__(kPrefixScanThreads)
adaptive_prefix_kernel(const float* score, int L, int32_t* start, float lo, float hi,
                       int advance, int32_t* len_out, float* tau_out, int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  __shared__ float warp_min[kPrefixScanThreads / 32];
  __shared__ float s_tau;
  __shared__ int s_fail[kPrefixScanThreads / 32], s_nan[kPrefixScanThreads / 32];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = __ldca(start + b);
  if (s < 0 || s > L) {
    if (tid == 0) {
      report(dev_status, DLLM_ERR_DEVICE_CHECK);
      len_out[b] = 0;
      tau_out[b] = INFINITY;
    }
    return;
  }
  const int A = L - s;
  if (A == 0) {
    if (tid == 0) {
      len_out[b] = 0;
      tau_out[b] = INFINITY;
    }
    return;
  }
  const float* row = score + (int64_t)b * L + s;
  const int seg = (A + kPrefixScanThreads - 1) / kPrefixScanThreads;
  const int p0 = tid * seg, p1 = min(A, p0 + seg);
  // 1. segment minimum (NaN counts as -inf) and first NaN
  float smin = INFINITY;
  int first_nan = A;
  for (int p = p0; p < p1; ++p) {
    const float v = __ldca(row + p);
    if (isnan(v)) {
      smin = -INFINITY;
      first_nan = min(first_nan, p);
    } else {
      smin = fminf(smin, v);
    }
  }
  // 2. exclusive block min-scan of the segment minima
  float incl = smin;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl = fminf(incl, t);
  }
  if (lane == 31) warp_min[warp] = incl;
  __syncthreads();
  float before_warp = INFINITY;
  for (int w = 0; w < warp; ++w) before_warp = fminf(before_warp, warp_min[w]);
  const float excl_lane = __shfl_up_sync(0xffffffffu, incl, 1);
  const float before = fminf(before_warp, lane == 0 ? INFINITY : excl_lane);
  // 3. tau = prefix minimum at k_lo
  // ceil(lo A) and floor(hi A) of the float32 fractions, products exact in double
  int k_lo = (int)ceil((double)lo * (double)A);
  k_lo = k_lo < 1 ? 1 : (k_lo > A ? A : k_lo);
  int k_hi = (int)floor((double)hi * (double)A);
  k_hi = k_hi < k_lo ? k_lo : k_hi;
  if (k_lo - 1 >= p0 && k_lo - 1 < p1) {
    float m = before;
    for (int p = p0; p < k_lo; ++p) {
      const float v = __ldca(row + p);
      m = fminf(m, isnan(v) ? -INFINITY : v);
    }
    s_tau = m;
  }
  __syncthreads();
  const float tau = s_tau;
  // 4. first position whose prefix minimum falls below tau
  int fail = A;
  {
    float m = before;
    for (int p = p0; p < p1; ++p) {
      const float v = __ldca(row + p);
      m = fminf(m, isnan(v) ? -INFINITY : v);
      if (!(m >= tau)) {
        fail = p;
        break;
      }
    }
  }
  fail = warp_min_int(fail);
  first_nan = warp_min_int(first_nan);
  if (lane == 0) {
    s_fail[warp] = fail;
    s_nan[warp] = first_nan;
  }
  __syncthreads();
  if (tid == 0) {
    int f = A, fn = A;
    for (int w = 0; w < kPrefixScanThreads / 32; ++w) {
      f = min(f, s_fail[w]);
      fn = min(fn, s_nan[w]);
    }
    int len = min(k_hi, min(f, fn));
    if (len < 1) len = 1;
    len_out[b] = len;
    tau_out[b] = tau;
    if (advance) start[b] = s + len;
  }
}

template <typename T>
int lock_nchunks(int V) {
  const int n = (V + lock_chunk_elems<T>() - 1) / lock_chunk_elems<T>();
  return n < 1 ? 1 : n;
}

template <typename T, bool CONF>
cudaError_t launch_lock_variant(const T* z, const T* y, int B, int R_src, int V, int64_t rs,
                                int64_t bs, int R_max, const int32_t* row_idx,
                                const int32_t* count, const int32_t* out_idx, int out_cols,
                                float eps, float gate_q, float* kl_out, float* unc_out,
                                float* conf_out, int32_t* argmax_out, float* margin_out,
                                uint8_t* locked, void* ws, int32_t* dev_status,
                                cudaStream_t stream) {
  constexpr int E = lvec<T>();
  const int nchunks = lock_nchunks<T>(V);
  if (nchunks > 65535 || (int64_t)B * R_max > INT_MAX) return cudaErrorInvalidConfiguration;
  const bool vec = (reinterpret_cast<uintptr_t>(z) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(y) % 16 == 0) && (rs % E == 0) && (bs % E == 0);
  LockPartial* part = static_cast<LockPartial*>(ws);
  // The partial kernels are launched after the previous kernel completes
  // (launch_serial), not with early residency: in the long-context step with
  // the confidence folded in (the partials right after the column sums), the
  // step took 662.7 us launched this way and 718.6 us with early residency.
  if (B <= kLockMaxB) {
    // persistent: DLLM_LOCK_MINB resident CTAs per SM over the valid items
    const int64_t items = (int64_t)B * R_max * nchunks;
    const int64_t cap = (int64_t)num_sms() * DLLM_LOCK_MINB;
    const int grid = (int)(items < cap ? items : cap);
    if (vec)
      launch_serial(lock_partial_persistent_kernel<T, true, CONF>, grid, kLockThreads, 0,
                    stream, z, y, R_src, V, rs, bs, B, R_max, row_idx, count, nchunks, part);
    else
      launch_serial(lock_partial_persistent_kernel<T, false, CONF>, grid, kLockThreads, 0,
                    stream, z, y, R_src, V, rs, bs, B, R_max, row_idx, count, nchunks, part);
  } else {
    dim3 grid(B * R_max, nchunks);
    if (vec)
      launch_serial(lock_partial_kernel<T, true, CONF>, grid, kLockThreads, 0, stream, z, y,
                    R_src, V, rs, bs, R_max, row_idx, count, nchunks, part);
    else
      launch_serial(lock_partial_kernel<T, false, CONF>, grid, kLockThreads, 0, stream, z, y,
                    R_src, V, rs, bs, R_max, row_idx, count, nchunks, part);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t rows = (int64_t)B * R_max;
  launch_pdl(lock_merge_kernel<CONF>, (unsigned)((rows + 7) / 8), 256, 0, stream, B, R_src,
             R_max, row_idx, count, out_idx, out_cols, nchunks, part, kl_out, unc_out, conf_out,
             argmax_out, margin_out, dev_status);
  e = cudaGetLastError();
  if (e != cudaSuccess || locked == nullptr) return e;
  const size_t smem = (size_t)R_max * sizeof(uint32_t);
  if (R_max > kGateMaxRows) return cudaErrorInvalidValue;
  // the limit is set once per kernel: raise it to the largest size any call uses
  e = ensure_smem_limit(reinterpret_cast<const void*>(lock_gate_kernel),
                        kGateMaxRows * (int)sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  launch_pdl(lock_gate_kernel, B, kGateThreads, smem, stream, R_max, count, out_idx, out_cols,
             kl_out, unc_out, eps, gate_q, locked, dev_status);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_lock_typed(const T* z, const T* y, int B, int R_src, int V, int64_t rs,
                              int64_t bs, int R_max, const int32_t* row_idx,
                              const int32_t* count, const int32_t* out_idx, int out_cols,
                              float eps, float gate_q, float* kl_out, float* unc_out,
                              float* conf_out, int32_t* argmax_out, float* margin_out,
                              uint8_t* locked, void* ws, int32_t* dev_status,
                              cudaStream_t stream) {
  if (conf_out != nullptr)
    return launch_lock_variant<T, true>(z, y, B, R_src, V, rs, bs, R_max, row_idx, count,
                                        out_idx, out_cols, eps, gate_q, kl_out, unc_out, conf_out,
                                        argmax_out, margin_out, locked, ws, dev_status, stream);
  return launch_lock_variant<T, false>(z, y, B, R_src, V, rs, bs, R_max, row_idx, count, out_idx,
                                       out_cols, eps, gate_q, kl_out, unc_out, nullptr, nullptr,
                                       nullptr, locked, ws, dev_status, stream);
}

}  // namespace

size_t lock_workspace_bytes(int B, int R_max, int V, int dtype) {
  const int n = dtype == DLLM_BF16 ? lock_nchunks<__nv_bfloat16>(V) : lock_nchunks<float>(V);
  return (size_t)B * (size_t)R_max * (size_t)n * sizeof(LockPartial);
}

cudaError_t launch_lock_criterion(const void* z, const void* y, int dtype, int B, int R_src,
                                  int V, int64_t rs, int64_t bs, int R_max,
                                  const int32_t* row_idx, const int32_t* count,
                                  const int32_t* out_idx, int out_cols, float eps, float gate_q,
                                  float* kl_out, float* unc_out, float* conf_out,
                                  int32_t* argmax_out, float* margin_out, uint8_t* locked,
                                  void* ws, int32_t* dev_status, cudaStream_t stream) {
  if (dtype == DLLM_BF16)
    return launch_lock_typed(static_cast<const __nv_bfloat16*>(z),
                             static_cast<const __nv_bfloat16*>(y), B, R_src, V, rs, bs, R_max,
                             row_idx, count, out_idx, out_cols, eps, gate_q, kl_out, unc_out,
                             conf_out, argmax_out, margin_out, locked, ws, dev_status, stream);
  return launch_lock_typed(static_cast<const float*>(z), static_cast<const float*>(y), B, R_src,
                           V, rs, bs, R_max, row_idx, count, out_idx, out_cols, eps, gate_q,
                           kl_out, unc_out, conf_out, argmax_out, margin_out, locked, ws,
                           dev_status, stream);
}

cudaError_t launch_adaptive_prefix(const float* score, int B, int L, int32_t* start, float lo,
                                   float hi, int advance_start, int32_t* len_out, float* tau_out,
                                   int32_t* dev_status, cudaStream_t stream) {
  launch_pdl(adaptive_prefix_kernel, B, kPrefixScanThreads, 0, stream, score, L, start, lo, hi,
             advance_start, len_out, tau_out, dev_status);
  return cudaGetLastError();
}

}  // namespace dllm
