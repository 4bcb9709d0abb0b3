// Partial attention (bf16, head dim 128) on the 5th-generation tensor cores.
//
// DyLLM ("Efficient Diffusion LLM Inference via Saliency-based Token Selection
// and Partial Attention"), technical summary, Methodology 2: the score rows of
// the salient queries are recomputed in full.  SureLock, technical summary
// section 2: active tokens attend to every position through the cached K/V,
// cost O(M N d).  Attn-Sampler, technical summary, Methodology 2: column sums
// of the attention matrix, computed block by block without materialising it.
//
// attn_fwd_tc_kernel -- one CTA per (128 active query rows, head, batch row):
//   warp 0     TMA producer: the Q tile once, then K/V tiles of 128 keys into
//              a two-stage ring (128-byte swizzle, 16 KB boxes of 64 dims).
//   warp 1     one thread issues tcgen05.mma: S = Q K^T into one of two TMEM
//              score buffers (so the next tile's QK^T overlaps the softmax),
//              then O += P V into a TMEM accumulator.
//   warps 2-5  softmax: each thread owns one query row (its TMEM lane), loads
//              the S row with tcgen05.ld, keeps a running maximum (rescaling O
//              in TMEM only when the maximum grows by more than 2^8) and sum,
//              and writes P in bf16 to shared memory in the operand layout the
//              P V product reads.  Epilogue: O / l in bf16 and the row's lse.
// attn_colsum_tc_kernel -- second normalised pass, one CTA per (128 keys,
//   head, batch row): S^T = K Q^T per tile of 128 active queries on the tensor
//   cores, then each thread (one key) adds exp(s - lse_i) over the active
//   rows.  Each key has one owner thread: no atomics, run-to-run identical.
//
// Every mbarrier wait is bounded (about a second); on expiry the kernel
// records DLLM_ERR_TIMEOUT in dev_status, drains its own copies and MMAs,
// frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace dllm {
namespace {

using namespace sm100;

constexpr int kBM = 128;       // query rows per tile
constexpr int kBN = 128;       // keys per tile
constexpr int kHD = 128;       // head dim
constexpr int kStages = 2;     // K/V (forward) or Q (column sums) ring depth
constexpr int kThreads = 192;  // 6 warps
constexpr uint32_t kBox = 16384;          // one 128-row x 64-dim bf16 box (swizzled)
constexpr uint32_t kTile = 2 * kBox;      // 128 rows x 128 dims
constexpr float kRescaleThreshold = 8.0f; // log2 units: P stays below 2^8

struct FwdParams {
  const int32_t* count;
  __nv_bfloat16* o;
  float* lse;
  int L, H, M_max;
  float scale_log2;
  int32_t* dev_status;
};

struct ColsumParams {
  const int32_t* count;
  const float* lse;
  float* colsum;
  int L, H, M_max;
  float scale_log2;
  int32_t* dev_status;
};

// shared-memory map of the forward kernel (offsets from a 1024-aligned base)
constexpr uint32_t kFwdQ = 0;
constexpr uint32_t kFwdK = kTile;                         // + s * 2 * kTile
constexpr uint32_t kFwdP = kTile + kStages * 2 * kTile;   // 160 KB
constexpr uint32_t kFwdBar = kFwdP + kTile;               // 192 KB
constexpr uint32_t kFwdSmem = kFwdBar + 256 + 1024;

// shared-memory map of the column-sum kernel
constexpr uint32_t kCsK = 0;
constexpr uint32_t kCsQ = kTile;                          // + s * kTile
constexpr uint32_t kCsLse = kTile + kStages * kTile;      // 2 x 128 floats
constexpr uint32_t kCsBar = kCsLse + 2 * kBM * 4;
constexpr uint32_t kCsSmem = kCsBar + 256 + 1024;

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Bounded wait whose outcome is the same for every lane of the warp (the
// tcgen05.ld/st that follow are warp-collective).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool r = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, r);
}

// Named barrier among the four softmax / epilogue warps (ids 2-5).
__device__ __forceinline__ void epi_bar_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, FwdParams p) {
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  int n = p.count[b];
  if (n < 0 || n > p.M_max) {
    if (qt == 0 && h == 0 && threadIdx.x == 0) report(p.dev_status, DLLM_ERR_DEVICE_CHECK);
    n = n < 0 ? 0 : p.M_max;
  }
  const int row0 = qt * kBM;
  if (row0 >= n) return;
  const int nkt = (p.L + kBN - 1) / kBN;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  const uint32_t sQ = base + kFwdQ, sP = base + kFwdP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kFwdBar);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [kStages]
  uint64_t* kv_empty = bars + 3;  // [kStages]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* s_free = bars + 7;    // [2]
  uint64_t* p_full = bars + 9;
  uint64_t* o_ready = bars + 10;
  uint64_t* mma_done = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  int* abort_flag = reinterpret_cast<int*>(bars + 13);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
    }
    mbar_init(p_full, 4);
    mbar_init(o_ready, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S0: +0, S1: +128, O: +256
  volatile int* abort = abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_expect_tx(q_full, kTile);
      tma_load_4d(gbase + kFwdQ, &tq, q_full, 0, h, row0, b);
      tma_load_4d(gbase + kFwdQ + kBox, &tq, q_full, 64, h, row0, b);
      int issued = 0;
      for (int it = 0; it < nkt; ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mbar_wait(&kv_empty[s], ((it / kStages) - 1) & 1, abort)) break;
        uint8_t* kdst = gbase + kFwdK + s * 2 * kTile;
        uint8_t* vdst = kdst + kTile;
        const int key0 = it * kBN;
        mbar_expect_tx(&kv_full[s], 2 * kTile);
        tma_load_4d(kdst, &tk, &kv_full[s], 0, h, key0, b);
        tma_load_4d(kdst + kBox, &tk, &kv_full[s], 64, h, key0, b);
        tma_load_4d(vdst, &tv, &kv_full[s], 0, h, key0, b);
        tma_load_4d(vdst + kBox, &tv, &kv_full[s], 64, h, key0, b);
        issued = it + 1;
      }
      // Drain: never leave with copies in flight into this CTA's shared memory.
      int none = 0;
      mbar_wait(q_full, 0, &none);
      for (int it = issued - kStages < 0 ? 0 : issued - kStages; it < issued; ++it)
        mbar_wait(&kv_full[it % kStages], (it / kStages) & 1, &none);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16_f32(kBM, kBN, false, false);
      const uint32_t id_pv = idesc_bf16_f32(kBM, kHD, false, true);
      bool ok = mbar_wait(q_full, 0, abort);
      auto issue_qk = [&](int it) -> bool {
        const int s = it % kStages, sb = it & 1;
        if (!mbar_wait(&kv_full[s], (it / kStages) & 1, abort)) return false;
        if (it >= 2 && !mbar_wait(&s_free[sb], ((it >> 1) - 1) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t sK = base + kFwdK + s * 2 * kTile;
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_bf16_ss(tmem + sb * kBN, smem_desc_sw128(sQ + off, 16, 1024),
                      smem_desc_sw128(sK + off, 16, 1024), id_qk, kk > 0);
        }
        mma_commit(&s_full[sb]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int it = 0; ok && it < nkt; ++it) {
        if (it + 1 < nkt && !issue_qk(it + 1)) break;
        if (!mbar_wait(p_full, it & 1, abort)) break;
        tc_fence_after();
        const int s = it % kStages;
        const uint32_t sV = base + kFwdK + s * 2 * kTile + kTile;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_bf16_ss(tmem + 2 * kBN, smem_desc_sw128(sP + aoff, 16, 1024),
                      smem_desc_sw128(sV + kk * 16 * 128, kBox, 1024), id_pv,
                      (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(o_ready);
        mma_commit(&kv_empty[s]);
      }
      // Every MMA issued above completes before the tensor memory is freed.
      mma_commit(mma_done);
      int none = 0;
      mbar_wait(mma_done, 0, &none);
    }
  } else {
    // ---------------------------------------------------------- softmax warps
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int it = 0; it < nkt; ++it) {
      const int sb = it & 1;
      if (!warp_wait(&s_full[sb], (it >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t raw[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c)
        tmem_ld_32x32b_x32(tmem + lane_base + sb * kBN + c * 32,
                           *reinterpret_cast<uint32_t(*)[32]>(&raw[c * 32]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);

      const int kvalid = min(kBN, p.L - it * kBN);
      float sv[kBN];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kBN; ++j) {
        const float s = (j < kvalid) ? __uint_as_float(raw[j]) * sl2 : -INFINITY;
        sv[j] = s;
        mx = fmaxf(mx, s);
      }
      const float m_new = fmaxf(m, mx);
      const bool grow = m_new > m + kRescaleThreshold;
      const float m_use = grow ? m_new : m;
      // P V of the previous tile must be done: the P buffer is reused and O
      // may be rescaled below.
      if (it > 0 && !warp_wait(o_ready, (it - 1) & 1, abort)) {
        ok = false;
        break;
      }
      if (grow) {
        const float alpha = ex2_approx(m - m_use);
        l *= alpha;
        if (it > 0) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kHD / 32; ++c) {
            uint32_t ov[32];
            tmem_ld_32x32b_x32(tmem + lane_base + 2 * kBN + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            tmem_st_32x32b_x32(tmem + lane_base + 2 * kBN + c * 32, ov);
          }
          tmem_st_wait();
        }
      }
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < kBN / 8; ++c) {
        float e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          e[k] = ex2_approx(sv[c * 8 + k] - m_use);
          sum += e[k];
        }
        const uint32_t addr = sP + (c >> 3) * kBox + r * 128 + ((((c & 7) ^ (r & 7))) << 4);
        st_shared_v4(addr, pack_bf16(e[0], e[1]), pack_bf16(e[2], e[3]), pack_bf16(e[4], e[5]),
                     pack_bf16(e[6], e[7]));
      }
      l += sum;
      m = m_use;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && warp_wait(o_ready, (nkt - 1) & 1, abort)) {
      tc_fence_after();
      const int i = row0 + r;
      const float inv = 1.0f / l;
      const bool store = i < n;
      __nv_bfloat16* orow = p.o + ((int64_t)b * p.M_max + i) * ((int64_t)p.H * kHD) + (int64_t)h * kHD;
#pragma unroll 1
      for (int c = 0; c < kHD / 32; ++c) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tmem + lane_base + 2 * kBN + c * 32, ov);
        tmem_ld_wait();
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(ov[v * 8 + 0]) * inv, __uint_as_float(ov[v * 8 + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(ov[v * 8 + 2]) * inv, __uint_as_float(ov[v * 8 + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(ov[v * 8 + 4]) * inv, __uint_as_float(ov[v * 8 + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(ov[v * 8 + 6]) * inv, __uint_as_float(ov[v * 8 + 7]) * inv);
            dst[v] = w;
          }
        }
      }
      if (store && p.lse != nullptr)
        p.lse[((int64_t)b * p.H + h) * p.M_max + i] = (m + log2f(l)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort) report(p.dev_status, DLLM_ERR_TIMEOUT);
}

__global__ void __launch_bounds__(kThreads, 1)
attn_colsum_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      ColsumParams p) {
  const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  int n = p.count[b];
  n = n < 0 ? 0 : (n > p.M_max ? p.M_max : n);
  const int nqt = (n + kBM - 1) / kBM;
  const int key0 = kt * kBN;
  float* out = p.colsum + ((int64_t)b * p.H + h) * p.L;
  if (nqt == 0) {
    for (int j = threadIdx.x; j < kBN; j += blockDim.x)
      if (key0 + j < p.L) out[key0 + j] = 0.f;
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  const uint32_t sK = base + kCsK;
  float* lse_s = reinterpret_cast<float*>(gbase + kCsLse);  // [2][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kCsBar);
  uint64_t* k_full = bars + 0;
  uint64_t* q_full = bars + 1;   // [kStages]
  uint64_t* q_empty = bars + 3;  // [kStages]
  uint64_t* s_full = bars + 5;   // [2]
  uint64_t* s_free = bars + 7;   // [2]
  uint64_t* mma_done = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  int* abort_flag = reinterpret_cast<int*>(bars + 11);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort = abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      mbar_expect_tx(k_full, kTile);
      tma_load_4d(gbase + kCsK, &tk, k_full, 0, h, key0, b);
      tma_load_4d(gbase + kCsK + kBox, &tk, k_full, 64, h, key0, b);
      int issued = 0;
      for (int it = 0; it < nqt; ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mbar_wait(&q_empty[s], ((it / kStages) - 1) & 1, abort)) break;
        uint8_t* qdst = gbase + kCsQ + s * kTile;
        mbar_expect_tx(&q_full[s], kTile);
        tma_load_4d(qdst, &tq, &q_full[s], 0, h, it * kBM, b);
        tma_load_4d(qdst + kBox, &tq, &q_full[s], 64, h, it * kBM, b);
        issued = it + 1;
      }
      int none = 0;
      mbar_wait(k_full, 0, &none);
      for (int it = issued - kStages < 0 ? 0 : issued - kStages; it < issued; ++it)
        mbar_wait(&q_full[it % kStages], (it / kStages) & 1, &none);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id = idesc_bf16_f32(kBN, kBM, false, false);
      bool ok = mbar_wait(k_full, 0, abort);
      for (int it = 0; ok && it < nqt; ++it) {
        const int s = it % kStages, sb = it & 1;
        if (!mbar_wait(&q_full[s], (it / kStages) & 1, abort)) break;
        if (it >= 2 && !mbar_wait(&s_free[sb], ((it >> 1) - 1) & 1, abort)) break;
        tc_fence_after();
        const uint32_t sQ = base + kCsQ + s * kTile;
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_bf16_ss(tmem + sb * kBM, smem_desc_sw128(sK + off, 16, 1024),
                      smem_desc_sw128(sQ + off, 16, 1024), id, kk > 0);
        }
        mma_commit(&s_full[sb]);
        mma_commit(&q_empty[s]);
      }
      mma_commit(mma_done);
      int none = 0;
      mbar_wait(mma_done, 0, &none);
    }
  } else {
    const int quarter = warp & 3;
    const int j = quarter * 32 + lane;  // key row of this thread
    const int t = threadIdx.x - 64;     // 0..127 for the lse loads
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float* lse_g = p.lse + ((int64_t)b * p.H + h) * p.M_max;
    const float sl2 = p.scale_log2;
    float acc = 0.f;
    bool ok = true;
    for (int it = 0; it < nqt; ++it) {
      // every epilogue thread passes the named barrier on every iteration,
      // also after an abort, so the barrier can never wait for a thread that left
      const int sb = it & 1;
      const int i = it * kBM + t;
      lse_s[sb * kBM + t] = i < n ? lse_g[i] * kLog2e : 0.f;
      epi_bar_sync();
      if (!ok) continue;
      if (!warp_wait(&s_full[sb], (it >> 1) & 1, abort)) {
        ok = false;
        continue;
      }
      tc_fence_after();
      uint32_t raw[kBM];
#pragma unroll
      for (int c = 0; c < kBM / 32; ++c)
        tmem_ld_32x32b_x32(tmem + lane_base + sb * kBM + c * 32,
                           *reinterpret_cast<uint32_t(*)[32]>(&raw[c * 32]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);
      const int nvalid = min(kBM, n - it * kBM);
      const float* ls = lse_s + sb * kBM;
#pragma unroll
      for (int q = 0; q < kBM; ++q) {
        const float e = ex2_approx(fmaf(__uint_as_float(raw[q]), sl2, -ls[q]));
        acc += (q < nvalid) ? e : 0.f;
      }
    }
    if (ok && key0 + j < p.L) out[key0 + j] = acc;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
  if (threadIdx.x == 0 && *abort) report(p.dev_status, DLLM_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [B, rows, H, 128] bf16 -> boxes of 64 dims x 128 rows (one head), 128-byte swizzle.
bool make_rows_map(CUtensorMap* map, const void* ptr, int B, int rows, int H) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kHD, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)kHD * 2, (cuuint64_t)H * kHD * 2,
                           (cuuint64_t)rows * H * kHD * 2};
  cuuint32_t box[4] = {64, 1, 128, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

bool attention_tc_supported(int dtype, int d, const void* q, const void* k, const void* v,
                            const void* o) {
  return dtype == DLLM_BF16 && d == kHD && reinterpret_cast<uintptr_t>(q) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(k) % 16 == 0 && reinterpret_cast<uintptr_t>(v) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(o) % 16 == 0 && encode_fn() != nullptr;
}

cudaError_t launch_attention_tc(const void* q, const void* k, const void* v, int B, int L, int H,
                                int M_max, const int32_t* count, float scale, void* o, float* lse,
                                float* colsum, int32_t* dev_status, cudaStream_t stream) {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kFwdSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(attn_colsum_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCsSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap tq, tk, tv;
  if (!make_rows_map(&tq, q, B, M_max, H) || !make_rows_map(&tk, k, B, L, H) ||
      !make_rows_map(&tv, v, B, L, H))
    return cudaErrorInvalidValue;
  FwdParams fp{count, static_cast<__nv_bfloat16*>(o), lse, L, H, M_max, scale * kLog2e, dev_status};
  dim3 grid((M_max + kBM - 1) / kBM, H, B);
  attn_fwd_tc_kernel<<<grid, kThreads, kFwdSmem, stream>>>(tq, tk, tv, fp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || colsum == nullptr) return e;
  ColsumParams cp{count, lse, colsum, L, H, M_max, scale * kLog2e, dev_status};
  dim3 cgrid((L + kBN - 1) / kBN, H, B);
  attn_colsum_tc_kernel<<<cgrid, kThreads, kCsSmem, stream>>>(tq, tk, cp);
  return cudaGetLastError();
}

}  // namespace dllm
