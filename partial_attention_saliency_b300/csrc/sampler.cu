// Attention-guided decoding order: total attention per position and the
// order and count of the tokens to decode.
//
// Attn-Sampler ("Attention-Based Sampler for Diffusion Language Models"),
// technical summary, Methodology 1: decoding in descending order of the
// column sums of the attention matrix; Methodology 2: tokens are decoded in
// parallel only while their score exceeds a threshold; the ablation on layers
// and heads: aggregate over all of them.
//
// attn_scores_kernel        one thread per (batch row, position): the sum
//                           over heads of the column sums, added in head
//                           order (optionally onto the scores of earlier
//                           layers); HBM bound, 4 H bytes read per position.
// attn_sampler_select_kernel one CTA per batch row: 64-bit keys
//                           (descending score, ascending position) of the
//                           candidates in shared memory, bitonic sort, the
//                           ordered positions, and the number of leading
//                           entries that reach the threshold.  The sort's
//                           stages with partners less than 64 keys apart run
//                           in registers, each warp on 64-key segments (two
//                           keys per lane, partners by warp shuffle); only the
//                           wider stages go through shared memory, one pair
//                           per thread and one CTA barrier each.
#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kSelectThreads = 1024;
constexpr int kSelectMaxL = 16384;  // 64-bit keys of a batch row in shared memory (128 KB)
constexpr int kSegKeys = 64;        // keys a warp sorts in registers (two per lane)

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kScoreThreads)
attn_scores_kernel(const float* colsum, int H, int L, int accumulate, float* score) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  const int b = blockIdx.y;
  const int j = blockIdx.x * kScoreThreads + threadIdx.x;
  if (j >= L) return;
  const float* c = colsum + (int64_t)b * H * L + j;
  float s = 0.f;
  for (int h = 0; h < H; ++h) s += __ldca(c + (int64_t)h * L);  // fixed head order
  float* out = score + (int64_t)b * L + j;
  *out = accumulate ? __ldca(out) + s : s;
}

// Key whose ascending order is descending score with equal scores by
// ascending position; -0 and +0 are equal, NaN sorts after every number.
__device__ __forceinline__ uint64_t order_key(float a, int pos) {
  uint32_t hi;
  if (isnan(a)) {
    hi = 0xffffffffu;
  } else {
    if (a == 0.f) a = 0.f;  // -0 -> +0
    const uint32_t u = __float_as_uint(a);
    const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    hi = ~asc;
  }
  return ((uint64_t)hi << 32) | (uint32_t)pos;
}

__global__ void __launch_bounds__(kSelectThreads)
attn_sampler_select_kernel(const float* score, int L, int N, const uint8_t* candidates, float tau,
                           float gamma, int k_max, int32_t* order, int32_t* n_out) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  extern __shared__ uint64_t keys[];  // [N], N a power of two >= L and >= 64
  __shared__ int s_cnt[kSelectThreads / 32], s_fail[kSelectThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* sc = score + (int64_t)b * L;
  const uint8_t* cd = candidates ? candidates + (int64_t)b * L : nullptr;
  // 1. keys of the candidates; everything else sorts last
  int cnt = 0;
  for (int j = tid; j < N; j += kSelectThreads) {
    uint64_t k = ~0ull;
    if (j < L && (cd == nullptr || __ldca(cd + j) != 0)) {
      k = order_key(__ldca(sc + j), j);
      ++cnt;
    }
    keys[j] = k;
  }
  cnt = warp_sum_int(cnt);
  if (lane == 0) s_cnt[warp] = cnt;
  __syncthreads();
  int n_cand = 0;
  for (int w = 0; w < kSelectThreads / 32; ++w) n_cand += s_cnt[w];
  // 2. bitonic sort, ascending.  Stage (k, j) orders each pair (i, i ^ j)
  // ascending where i & k is 0 and descending elsewhere.
  // The stages j = min(k, 64) / 2 .. 1 of every k <= N, in registers: lane
  // l of a warp holds keys base + 2l and base + 2l + 1 of a 64-key segment.
  auto register_stages = [&](int k_lo, int k_hi) {
    for (int base = warp * kSegKeys; base < N; base += kSelectThreads / 32 * kSegKeys) {
      const int i0 = base + 2 * lane;
      uint64_t a = keys[i0], c = keys[i0 + 1];
      for (int k = k_lo; k <= k_hi; k <<= 1) {
        const bool up = (i0 & k) == 0;
        for (int j = (k < kSegKeys ? k : kSegKeys) >> 1; j > 1; j >>= 1) {
          const uint64_t pa = __shfl_xor_sync(0xffffffffu, a, j >> 1);
          const uint64_t pc = __shfl_xor_sync(0xffffffffu, c, j >> 1);
          const bool keep_min = ((lane & (j >> 1)) == 0) == up;  // lower of the pair, ascending
          a = keep_min ? (a < pa ? a : pa) : (a > pa ? a : pa);
          c = keep_min ? (c < pc ? c : pc) : (c > pc ? c : pc);
        }
        if ((a > c) == up) {  // j = 1: the lane's own two keys
          const uint64_t x = a;
          a = c;
          c = x;
        }
      }
      keys[i0] = a;
      keys[i0 + 1] = c;
    }
    __syncthreads();
  };
  register_stages(2, kSegKeys);
  for (int k = 2 * kSegKeys; k <= N; k <<= 1) {
    // the stages with partners at least 64 keys apart: pair p of N / 2 is
    // (i, i + j), i the index p with a zero bit inserted at j
    for (int j = k >> 1; j >= kSegKeys; j >>= 1) {
      for (int p = tid; p < N / 2; p += kSelectThreads) {
        const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1)), ixj = i | j;
        const uint64_t x = keys[i], y = keys[ixj];
        if ((x > y) == ((i & k) == 0)) {
          keys[i] = y;
          keys[ixj] = x;
        }
      }
      __syncthreads();
    }
    register_stages(k, k);
  }
  // 3. the ordered positions, and the first entry below the threshold
  float thr = tau;
  if (n_cand > 0 && gamma > 0.f) {
    const float top = __ldca(sc + (int)(uint32_t)keys[0]);
    thr = fmaxf(tau, __fmul_rn(gamma, top));  // a NaN top leaves tau
  }
  int fail = n_cand;
  int32_t* ob = order + (int64_t)b * L;
  for (int i = tid; i < L; i += kSelectThreads) {
    if (i < n_cand) {
      const int pos = (int)(uint32_t)keys[i];
      ob[i] = pos;
      if (!(__ldca(sc + pos) >= thr) && i < fail) fail = i;
    } else {
      ob[i] = -1;
    }
  }
  fail = warp_min_int(fail);
  if (lane == 0) s_fail[warp] = fail;
  __syncthreads();
  if (tid == 0) {
    int n = n_cand;
    for (int w = 0; w < kSelectThreads / 32; ++w) n = min(n, s_fail[w]);
    if (k_max > 0) n = min(n, k_max);
    if (n_cand > 0 && n < 1) n = 1;
    n_out[b] = n;
  }
}

}  // namespace

cudaError_t launch_attn_scores(const float* colsum, int B, int H, int L, int accumulate,
                               float* score, cudaStream_t stream) {
  const dim3 grid((unsigned)((L + kScoreThreads - 1) / kScoreThreads), (unsigned)B);
  launch_pdl(attn_scores_kernel, grid, kScoreThreads, 0, stream, colsum, H, L, accumulate, score);
  return cudaGetLastError();
}

int attn_sampler_max_len() { return kSelectMaxL; }

cudaError_t launch_attn_sampler_select(const float* score, int B, int L,
                                       const uint8_t* candidates, float tau, float gamma,
                                       int k_max, int32_t* order, int32_t* n_out,
                                       cudaStream_t stream) {
  if (L < 1 || L > kSelectMaxL) return cudaErrorInvalidValue;
  int N = kSegKeys;
  while (N < L) N <<= 1;
  // the limit is set once per kernel: raise it to the largest size any call uses
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(attn_sampler_select_kernel),
                                    kSelectMaxL * (int)sizeof(uint64_t));
  if (e != cudaSuccess) return e;
  launch_pdl(attn_sampler_select_kernel, B, kSelectThreads, (size_t)N * sizeof(uint64_t), stream,
             score, L, N, candidates, tau, gamma, k_max, order, n_out);
  return cudaGetLastError();
}

}  // namespace dllm
