// Partial attention (bf16, head dim 128) on the 5th-generation tensor cores.
//
// DyLLM ("Efficient Diffusion LLM Inference via Saliency-based Token Selection
// and Partial Attention"), technical summary, Methodology 2: the score rows of
// the salient queries are recomputed in full.  SureLock, technical summary
// section 2: active tokens attend to every position through the cached K/V,
// cost O(M N d).  Attn-Sampler, technical summary, Methodology 2: column sums
// of the attention matrix, computed block by block without materialising it.
//
// attn_fwd_tc_kernel -- persistent, one CTA per SM; a work item is a pair of
//   query tiles of 128 active rows of one (batch row, head), or a single tile
//   when the head has an odd number of tiles, optionally limited to a slice
//   of the key range when there are too few items for the SMs
//   (attn_split_merge_kernel then combines the slices):
//   warp 8     TMA producer: the Q tiles once per item, then K and V tiles of
//              128 keys into a three-stage K ring and a two-stage V ring
//              (128-byte swizzle, 16 KB boxes of 64 dims).
//   warp 9     one thread issues tcgen05.mma: S_x = Q K^T into one of two TMEM
//              score buffers, then O_x += P_x V into a TMEM accumulator.
//   warps 0-7  two softmax warpgroups, slot x = warp / 4, each thread one
//              query row (its TMEM lane).  In a pair item slot x holds query
//              tile x over every key tile (the two tiles ping-pong on the
//              tensor cores and share each K/V tile).  In a one-tile item slot
//              x takes the key tiles t with t % 2 == x, so the next tile's
//              Q K^T never waits for this tile's softmax, and slot 0 merges
//              slot 1's partial O, maximum and sum at the end.  Each slot
//              loads its S row with tcgen05.ld, keeps a running maximum
//              (rescaling O in TMEM only when it grows by more than 2^8) and
//              sum, and writes P in bf16 back over S, where the P V product
//              reads it.  Epilogue: O / l in bf16 and the row's lse.
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
constexpr uint32_t kBox = 16384;          // one 128-row x 64-dim bf16 box (swizzled)
constexpr uint32_t kTile = 2 * kBox;      // 128 rows x 128 dims
constexpr float kRescaleThreshold = 8.0f; // log2 units: P stays below 2^8

// Forward kernel roles: warps 0-3 softmax of query tile A, warps 4-7 softmax
// of query tile B (warp w reads TMEM lanes 32 * (w % 4) .. + 31), warp 8 TMA
// producer, warp 9 MMA issuer.
constexpr int kFwdThreads = 320;
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
// Exponential pairs computed on the FMA pipe (exp2_poly2) instead of MUFU,
// out of every 8: the forward softmax is otherwise bound by the MUFU ex2
// rate.  The column sums are not (measured faster with MUFU alone: their
// FMA pipe is busy with the scaling and the sums).
constexpr int kFwdPoly = 2;
constexpr int kColsumPoly = 0;       // persistent column-sum kernel
constexpr int kColsumGroupPoly = 0;  // key-tile-group kernel (2 or 3 of 8 measured slower)

struct FwdParams {
  const int32_t* count;
  __nv_bfloat16* o;
  float* lse;
  float* ws_o;   // split partials: [item][2 tiles][128 rows][128 dims] unnormalised O
  float* ws_ml;  // split partials: [item][2 tiles][128 rows][2] = (max (log2 units), sum)
  int B, L, H, M_max;
  int max_split_items;  // capacity of the workspace in items (0: never split)
  float scale_log2;
  int32_t* dev_status;
  long long wait_limit;  // clock cycles a pipeline wait may take (drains excepted)
};

struct ColsumParams {
  const int32_t* count;
  const float* lse;
  float* colsum;
  int L, H, M_max;
  float scale_log2;
  int32_t* dev_status;
  int min_qt;  // the kernel handles batch rows with more than min_qt - 1 query tiles
};

// Batch rows with at most kCsMaxQt query tiles (and empty rows) take the
// persistent column-sum kernel; the others the key-tile-group kernel.
constexpr int kCsMaxQt = 2;

// Key tiles of 128 below which the forward never splits the key range.
constexpr int kMinSplitTiles = 12;

// shared-memory map of the forward kernel (offsets from a 1024-aligned base).
// K and V have rings of their own: a K tile is free once the Q K^T products
// of its tile are done, a V tile only after the P V products, so K runs a
// stage deeper and its loads start earlier.
constexpr int kKStages = 3;                                // K ring depth
constexpr int kVStages = 2;                                // V ring depth
constexpr uint32_t kFwdQ = 0;                              // Q tile A, then Q tile B
constexpr uint32_t kFwdK = 2 * kTile;                      // + s * kTile
constexpr uint32_t kFwdV = kFwdK + kKStages * kTile;       // + s * kTile
constexpr uint32_t kFwdBar = kFwdV + kVStages * kTile;     // 224 KB
constexpr uint32_t kFwdX = kFwdBar + 256;                  // one-tile items: (m, l) of slot 1
constexpr uint32_t kFwdSmem = kFwdX + 2 * kBM * 4 + 1024;

// tensor-memory columns of the forward kernel (512 allocated): scores S of
// tile A and B (P overwrites the first 64 columns of its S as bf16 pairs),
// then the O accumulators of A and B
constexpr uint32_t kTmS = 0;     // + X * 128
constexpr uint32_t kTmO = 256;   // + X * 128


__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Bounded wait whose outcome is the same for every lane of the warp (the
// tcgen05.ld/st that follow are warp-collective).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          long long limit = kWaitLimitDefault) {
  const bool r = mbar_wait(bar, parity, abort, limit);
  return __all_sync(0xffffffffu, r);
}


// Work plan shared by the forward and merge kernels, computed on the device
// from the active counts.  A work item is a pair of query tiles of 128
// active rows (tile A, and tile B when the head has one more tile) of one
// (batch row, head), optionally limited to a slice of the key range.  The
// pairs are dealt round-robin to the persistent CTAs; the pairs of the last,
// partly filled round (all pairs when there are fewer pairs than CTAs) are
// split over the key range so that the round keeps every SM busy, and a
// merge kernel combines their slices.
struct FwdPlan {
  int total_qp;  // tile pairs over all (b, h)
  int n_full;    // pairs [0, n_full) are one item each over all keys
  int nsplit;    // key-range splits of each pair in [n_full, total_qp)
  int tps;       // key tiles per split
  int nkt;       // key tiles of the sequence
};

__device__ __forceinline__ int clamp_count(const int32_t* count, int b, int M_max) {
  const int n = __ldca(count + b);
  return n < 0 ? 0 : (n > M_max ? M_max : n);
}

__device__ __forceinline__ int pairs_of(int n) { return (((n + kBM - 1) / kBM) + 1) / 2; }

// Clamped active counts of the first kPlanMaxB batch rows, staged in shared
// memory once per CTA (the plan is decoded for every work item); rows beyond
// are read from global memory.
constexpr int kPlanMaxB = 64;

__device__ __forceinline__ int cnt_of(const FwdParams& p, const int* s_cnt, int b) {
  return b < kPlanMaxB ? s_cnt[b] : clamp_count(p.count, b, p.M_max);
}

__device__ __forceinline__ void stage_counts(const FwdParams& p, int* s_cnt) {
  for (int b = threadIdx.x; b < p.B && b < kPlanMaxB; b += blockDim.x)
    s_cnt[b] = clamp_count(p.count, b, p.M_max);
}

__device__ FwdPlan make_plan(const FwdParams& p, const int* s_cnt, int n_ctas) {
  FwdPlan pl;
  pl.nkt = (p.L + kBN - 1) / kBN;
  int qp = 0;
  for (int b = 0; b < p.B; ++b) qp += p.H * pairs_of(cnt_of(p, s_cnt, b));
  pl.total_qp = qp;
  int ns = 1, tail = 0;
  if (qp > 0 && p.max_split_items > 0) {
    if (qp < n_ctas) {
      // as many splits as fit in one round: with at least half the SMs busy
      // (ns = 1) every SM streams its pair's whole key range and no merge is
      // needed; the HBM, not the SM count, is then the limit
      tail = qp;
      ns = n_ctas / qp;
    } else if (2 * (qp % n_ctas) <= n_ctas) {  // a last round at most half full
      tail = qp % n_ctas;
      ns = tail > 0 ? n_ctas / tail : 1;
    }
    const int max_by_tiles = pl.nkt / 2 > 1 ? pl.nkt / 2 : 1;  // at least two key tiles each
    ns = ns < max_by_tiles ? ns : max_by_tiles;
    if (tail > 0) {
      const int max_by_ws = p.max_split_items / tail;
      ns = ns < max_by_ws ? ns : max_by_ws;
    }
    if (ns < 1) ns = 1;
  }
  pl.tps = (pl.nkt + ns - 1) / ns;
  pl.nsplit = (pl.nkt + pl.tps - 1) / pl.tps;  // no empty split
  pl.n_full = pl.nsplit > 1 ? qp - tail : qp;
  return pl;
}

__device__ __forceinline__ int plan_items(const FwdPlan& pl) {
  return pl.n_full + (pl.total_qp - pl.n_full) * pl.nsplit;
}

// Work item v -> (pair index, first key tile, key tiles, split slot or -1).
__device__ __forceinline__ void item_of(const FwdPlan& pl, int v, int* qi, int* kt0, int* nt,
                                        int* slot) {
  if (v < pl.n_full) {
    *qi = v;
    *kt0 = 0;
    *nt = pl.nkt;
    *slot = -1;
  } else {
    const int u = v - pl.n_full;
    const int split = u % pl.nsplit;
    *qi = pl.n_full + u / pl.nsplit;
    *kt0 = split * pl.tps;
    *nt = min(pl.tps, pl.nkt - *kt0);
    *slot = u;
  }
}

// Pair index qi -> (b, h, pair, query tiles in the pair), batch-major then
// head-major.
__device__ __forceinline__ void decode_pair(const FwdParams& p, const int* s_cnt, int qi, int* b,
                                            int* h, int* pair, int* nq) {
  for (int bb = 0; bb < p.B; ++bb) {
    const int n = cnt_of(p, s_cnt, bb);
    const int nqt = (n + kBM - 1) / kBM;
    const int per_head = (nqt + 1) / 2;
    if (qi < per_head * p.H) {
      *b = bb;
      *h = qi / per_head;
      *pair = qi - *h * per_head;
      *nq = min(2, nqt - 2 * *pair);
      return;
    }
    qi -= per_head * p.H;
  }
  *b = *h = *pair = 0;
  *nq = 0;
}

// Persistent forward kernel: one CTA per SM walks the work items round-robin.
// Per key tile t the MMA warp issues, in this order,
//   O_A += P_A(t) V(t),  S_A = Q_A K(t+1)^T,  O_B += P_B(t) V(t),  S_B = Q_B K(t+1)^T
// so that the tensor cores work on one tile while the softmax warps of the
// other tile compute its probabilities.  P overwrites the S it came from in
// tensor memory and feeds the P V product from there.  Because tcgen05
// operations of one thread complete in issue order, "S_X(t+1) is full"
// also means O_X += P_X(t) V(t) has completed, so the softmax warps may
// rescale O_X in place when their running maximum grows.
__global__ void __launch_bounds__(kFwdThreads, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, FwdParams p) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kFwdBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;    // [kKStages]
  uint64_t* k_empty = bars + 5;   // [kKStages]
  uint64_t* v_full = bars + 8;    // [kVStages]
  uint64_t* v_empty = bars + 10;  // [kVStages]
  uint64_t* s_full = bars + 12;   // [2]: S of tile A / B written
  uint64_t* p_full = bars + 14;   // [2]: P of tile A / B written (4 warps each)
  uint64_t* o_done = bars + 16;   // [2]: last P V of the item completed
  uint64_t* o_free = bars + 18;   // [2]: epilogue has read O (4 warps each)
  uint64_t* mma_done = bars + 20;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 21);
  int* abort_flag = reinterpret_cast<int*>(bars + 22);
  uint64_t* x_ready = bars + 23;  // one-tile items: slot 1's (m, l) published (4 warps)
  float* x_ml = reinterpret_cast<float*>(gbase + kFwdX);  // [2][128]: m, then l

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 4);
      mbar_init(&o_done[x], 1);
      mbar_init(&o_free[x], 4);
    }
    mbar_init(mma_done, 1);
    mbar_init(x_ready, 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpTma) tmem_alloc(tmem_slot, 512);
  __shared__ int s_cnt[kPlanMaxB];
  stage_counts(p, s_cnt);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    for (int b = 0; b < p.B; ++b) {
      const int c = __ldca(p.count + b);
      if (c < 0 || c > p.M_max) report(p.dev_status, DLLM_ERR_DEVICE_CHECK);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort = abort_flag;
  const FwdPlan plan = make_plan(p, s_cnt, gridDim.x);
  const int n_items = plan_items(plan);
  if ((int)blockIdx.x >= n_items) {  // no work: give the tensor memory back
    if (warp == kWarpTma) tmem_dealloc(tmem, 512);
    return;
  }

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // keys stay in L2 for the column-sum pass that reads them next; values
      // are read once
      const uint64_t pol_k = l2_policy_evict_last();
      const uint64_t pol_v = l2_policy_evict_first();
      int j = 0, gk = 0, gv = 0;  // items, K tiles and V tiles issued
      bool ok = true;
      for (int v = blockIdx.x; ok && v < n_items; v += gridDim.x, ++j) {
        int b, h, pair, nq, qi, kt0, nt, slot;
        item_of(plan, v, &qi, &kt0, &nt, &slot);
        decode_pair(p, s_cnt, qi, &b, &h, &pair, &nq);
        if (j > 0 && !mbar_wait(q_empty, (j - 1) & 1, abort, p.wait_limit)) break;
        mbar_expect_tx(q_full, (uint32_t)nq * kTile);
        for (int x = 0; x < nq; ++x) {
          const int row0 = (2 * pair + x) * kBM;
          tma_load_4d(gbase + kFwdQ + x * kTile, &tq, q_full, 0, h, row0, b);
          tma_load_4d(gbase + kFwdQ + x * kTile + kBox, &tq, q_full, 64, h, row0, b);
        }
        // K(t), then V(t): V(t)'s slot is freed by the P V products of tile
        // t - 2, which also lets K(t + 1) start three tiles before its Q K^T.
        for (int t = 0; t < nt; ++t) {
          const int key0 = (kt0 + t) * kBN;
          const int sk = gk % kKStages;
          if (gk >= kKStages && !mbar_wait(&k_empty[sk], ((gk / kKStages) - 1) & 1, abort, p.wait_limit)) {
            ok = false;
            break;
          }
          uint8_t* kdst = gbase + kFwdK + sk * kTile;
          mbar_expect_tx(&k_full[sk], kTile);
          tma_load_4d_hint(kdst, &tk, &k_full[sk], 0, h, key0, b, pol_k);
          tma_load_4d_hint(kdst + kBox, &tk, &k_full[sk], 64, h, key0, b, pol_k);
          ++gk;
          const int sv = gv % kVStages;
          if (gv >= kVStages && !mbar_wait(&v_empty[sv], ((gv / kVStages) - 1) & 1, abort, p.wait_limit)) {
            ok = false;
            break;
          }
          uint8_t* vdst = gbase + kFwdV + sv * kTile;
          mbar_expect_tx(&v_full[sv], kTile);
          tma_load_4d_hint(vdst, &tv, &v_full[sv], 0, h, key0, b, pol_v);
          tma_load_4d_hint(vdst + kBox, &tv, &v_full[sv], 64, h, key0, b, pol_v);
          ++gv;
        }
      }
      // Drain: never leave with copies in flight into this CTA's shared memory.
      int none = 0;
      if (j > 0) mbar_wait(q_full, (j - 1) & 1, &none);
      for (int k = gk - kKStages < 0 ? 0 : gk - kKStages; k < gk; ++k)
        mbar_wait(&k_full[k % kKStages], (k / kKStages) & 1, &none);
      for (int k = gv - kVStages < 0 ? 0 : gv - kVStages; k < gv; ++k)
        mbar_wait(&v_full[k % kVStages], (k / kVStages) & 1, &none);
      if (none) report(p.dev_status, DLLM_ERR_TIMEOUT);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16_f32(kBM, kBN, false, false);
      const uint32_t id_pv = idesc_bf16_f32(kBM, kHD, false, true);
      // S_x = Q_qx K(s)^T, then s_full[x]
      auto issue_qk = [&](int qx, int x, int s) {
        const uint32_t sQ = base + kFwdQ + qx * kTile;
        const uint32_t sK = base + kFwdK + s * kTile;
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_bf16_ss(tmem + kTmS + x * kBN, smem_desc_sw128(sQ + off, 16, 1024),
                      smem_desc_sw128(sK + off, 16, 1024), id_qk, kk > 0);
        }
        mma_commit(&s_full[x]);
      };
      auto issue_pv = [&](int x, int s, bool acc) {
        const uint32_t sV = base + kFwdV + s * kTile;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_bf16_ts(tmem + kTmO + x * kHD, tmem + kTmS + x * kBN + kk * 8,
                      smem_desc_sw128(sV + kk * 16 * 128, kBox, 1024), id_pv,
                      (acc || kk > 0) ? 1u : 0u);
      };
      int j = 0, g = 0;          // items, K/V tiles
      int gt[2] = {0, 0};        // tiles processed per query tile slot
      int jt[2] = {0, 0};        // items processed per query tile slot
      bool ok = true;
      for (int v = blockIdx.x; ok && v < n_items; v += gridDim.x, ++j) {
        int b, h, pair, nq, qi, kt0, nt, slot;
        item_of(plan, v, &qi, &kt0, &nt, &slot);
        decode_pair(p, s_cnt, qi, &b, &h, &pair, &nq);
        if (!mbar_wait(q_full, j & 1, abort, p.wait_limit)) break;
        if (nq == 2) {
          // Pair of query tiles: per key tile t the order is
          //   O_A += P_A(t) V(t), S_A = Q_A K(t+1)^T, O_B += P_B(t) V(t), S_B = Q_B K(t+1)^T.
          if (!mbar_wait(&k_full[g % kKStages], (g / kKStages) & 1, abort, p.wait_limit)) break;
          tc_fence_after();
          for (int x = 0; x < 2; ++x) issue_qk(x, x, g % kKStages);
          mma_commit(&k_empty[g % kKStages]);  // K(0) is read by its Q K^T products only
          if (nt == 1) mma_commit(q_empty);
          for (int t = 0; t < nt && ok; ++t) {
            const int sv = (g + t) % kVStages;
            const int sk1 = (g + t + 1) % kKStages;
            const bool more = t + 1 < nt;
            for (int x = 0; x < 2; ++x) {
              if (!mbar_wait(&p_full[x], gt[x] & 1, abort, p.wait_limit)) {
                ok = false;
                break;
              }
              if (t == 0 && jt[x] > 0 && !mbar_wait(&o_free[x], (jt[x] - 1) & 1, abort, p.wait_limit)) {
                ok = false;
                break;
              }
              if (x == 0 && !mbar_wait(&v_full[sv], ((g + t) / kVStages) & 1, abort, p.wait_limit)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_pv(x, sv, t > 0);
              if (x == 1) mma_commit(&v_empty[sv]);  // V(t) no longer read
              if (more) {
                if (x == 0 && !mbar_wait(&k_full[sk1], ((g + t + 1) / kKStages) & 1, abort, p.wait_limit)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                issue_qk(x, x, sk1);
                if (x == 1) {
                  mma_commit(&k_empty[sk1]);                // K(t + 1) no longer read
                  if (t + 2 == nt) mma_commit(q_empty);     // last read of Q
                }
              } else {
                mma_commit(&o_done[x]);
              }
              ++gt[x];
            }
          }
          g += nt;
          ++jt[0];
          ++jt[1];
        } else {
          // One query tile: key tile t goes to slot x = t % 2 (S_x, then
          // O_x), so the two softmax warpgroups take alternate key tiles and
          // the Q K^T of tile t + 2 is issued right after the P V of tile t.
          for (int t = 0; t < 2 && t < nt && ok; ++t) {
            const int sk = (g + t) % kKStages;
            if (!mbar_wait(&k_full[sk], ((g + t) / kKStages) & 1, abort, p.wait_limit)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_qk(0, t, sk);
            mma_commit(&k_empty[sk]);
          }
          if (ok && nt <= 2) mma_commit(q_empty);
          for (int t = 0; t < nt && ok; ++t) {
            const int x = t & 1;
            const int sv = (g + t) % kVStages;
            if (!mbar_wait(&p_full[x], gt[x] & 1, abort, p.wait_limit)) {
              ok = false;
              break;
            }
            if (t < 2 && jt[x] > 0 && !mbar_wait(&o_free[x], (jt[x] - 1) & 1, abort, p.wait_limit)) {
              ok = false;
              break;
            }
            if (!mbar_wait(&v_full[sv], ((g + t) / kVStages) & 1, abort, p.wait_limit)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(x, sv, t >= 2);
            mma_commit(&v_empty[sv]);  // V(t) no longer read
            if (t + 2 < nt) {
              const int sk = (g + t + 2) % kKStages;
              if (!mbar_wait(&k_full[sk], ((g + t + 2) / kKStages) & 1, abort, p.wait_limit)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_qk(0, x, sk);
              mma_commit(&k_empty[sk]);
              if (t + 3 == nt) mma_commit(q_empty);  // last read of Q
            } else {
              mma_commit(&o_done[x]);
            }
            ++gt[x];
          }
          g += nt;
          ++jt[0];
          if (nt > 1) ++jt[1];
        }
      }
      // Every MMA issued above completes before the tensor memory is freed.
      mma_commit(mma_done);
      int none = 0;
      mbar_wait(mma_done, 0, &none);
      if (none) report(p.dev_status, DLLM_ERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    // Slot x = warp / 4 owns S_x and O_x.  In a pair item slot x holds query
    // tile x over every key tile; in a one-tile item both slots hold the same
    // query tile, slot x the key tiles t with t % 2 == x, and slot 0 merges
    // slot 1's partial O, maximum and sum into the result.
    const int x = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row of the tile
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + kTmS + x * kBN;
    const uint32_t tO = tmem + lane_base + kTmO + x * kHD;
    const uint32_t tO1 = tmem + lane_base + kTmO + kHD;  // slot 1's O (read by slot 0)
    const float sl2 = p.scale_log2;
    int gx = 0, jx = 0, jd = 0;  // tiles and items of this slot, merged one-tile items
    bool ok = true;
    for (int v = blockIdx.x; ok && v < n_items; v += gridDim.x) {
      int b, h, pair, nq, qi, kt0, nt, wslot;
      item_of(plan, v, &qi, &kt0, &nt, &wslot);
      decode_pair(p, s_cnt, qi, &b, &h, &pair, &nq);
      const bool single = nq == 1;
      const int qtile = single ? 0 : x;  // query tile of the pair this slot reads
      const int mine = single ? (x == 0 ? (nt + 1) / 2 : nt / 2) : nt;  // key tiles of this slot
      if (mine == 0) continue;
      const bool merge = single && nt > 1;  // slot 0 combines both slots' results
      // A warp whose 32 rows all lie past the count only keeps the
      // handshakes: its P rows feed only O rows that are never stored (row i
      // of P V depends on row i of P alone).
      const bool idle = (2 * pair + qtile) * kBM + quarter * 32 >= cnt_of(p, s_cnt, b);
      float m = -INFINITY, l = 0.f;
      // key tiles kt0 + x, kt0 + x + 2, ... (one-tile item) or kt0, kt0 + 1, ...
      const int kstep = single ? 2 : 1;
      int kvalid = p.L - (kt0 + (single ? x : 0)) * kBN;  // < kBN only on the last, partial tile
      for (int tt = 0; tt < mine; ++tt, ++gx, kvalid -= kstep * kBN) {
        if (!warp_wait(&s_full[x], gx & 1, abort, p.wait_limit)) {
          ok = false;
          break;
        }
        if (idle) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[x]);
          continue;
        }
        tc_fence_after();
        // The whole S row (128 keys) is read with one wait; the row maximum
        // is a 4-way tree; P = 2^(s * scale * log2 e - m) is then produced
        // in chunks of 32 keys and stored as bf16 pairs into the first 64
        // columns of S (P column j holds keys 2j, 2j + 1; those S columns
        // are already in registers).
        uint32_t raw[kBN];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c)
          tmem_ld_32x32b_x32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&raw[c * 32]));
        tmem_ld_wait();
        if (kvalid < kBN) {  // warp-uniform
#pragma unroll
          for (int q = 0; q < kBN; ++q)
            if (q >= kvalid) raw[q] = 0xff800000u;  // -inf
        }
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < kBN; q += 8)
          mx4[(q >> 3) & 3] =
              fmax3(mx4[(q >> 3) & 3],
                    fmax3(__uint_as_float(raw[q]), __uint_as_float(raw[q + 1]),
                          __uint_as_float(raw[q + 2])),
                    fmax3(__uint_as_float(raw[q + 3]),
                          fmax3(__uint_as_float(raw[q + 4]), __uint_as_float(raw[q + 5]),
                                __uint_as_float(raw[q + 6])),
                          __uint_as_float(raw[q + 7])));
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        const float m_new = fmaxf(m, mx * sl2);
        const bool grow = m_new > m + kRescaleThreshold;
        const float alpha = grow ? ex2_approx(m - m_new) : 1.0f;
        if (grow) {
          l *= alpha;
          m = m_new;
        }
        const float2 sl2x2 = make_float2(sl2, sl2);
        const float2 negm = make_float2(-m, -m);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) {
            const int q = c * 32 + cc * 2;
            const float2 a2 = __ffma2_rn(
                make_float2(__uint_as_float(raw[q]), __uint_as_float(raw[q + 1])), sl2x2, negm);
            float2 e;
            if ((cc & 7) >= 8 - kFwdPoly) {
              e = exp2_poly2(a2);
            } else {
              e.x = ex2_approx(a2.x);
              e.y = ex2_approx(a2.y);
            }
            if (cc & 1)
              acc1 = __fadd2_rn(acc1, e);
            else
              acc0 = __fadd2_rn(acc0, e);
            pk[cc] = pack_bf16(e.x, e.y);
          }
          tmem_st_32x32b_x16(tS + c * 16, pk);
        }
        // O is rescaled in place when some row's maximum grew (tcgen05.ld/st
        // are warp-collective, so the warp votes; rows that did not grow
        // multiply by 1).  The slot's first P V of an item is written without
        // accumulation and needs none.
        if (tt > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int c = 0; c < kHD / 32; ++c) {
            uint32_t ov[32];
            tmem_ld_32x32b_x32(tO + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) ov[q] = __float_as_uint(__uint_as_float(ov[q]) * alpha);
            tmem_st_32x32b_x32(tO + c * 32, ov);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x]);
        l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
      }
      if (!ok || !warp_wait(&o_done[x], jx & 1, abort, p.wait_limit)) {
        ok = false;
        break;
      }
      ++jx;
      if (merge && x == 1) {
        // slot 1 publishes its maximum and sum; slot 0 reads O_1 and
        // releases it
        if (!idle) {
          x_ml[r] = m;
          x_ml[kBM + r] = l;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(x_ready);
        continue;
      }
      // ---------------------------------------------------------- epilogue
      float a0 = 1.0f, a1 = 0.0f;  // weights of O_x and O_1 (merged one-tile items)
      if (merge) {
        if (!warp_wait(x_ready, jd & 1, abort, p.wait_limit)) {
          ok = false;
          break;
        }
        ++jd;
        if (!idle) {
          const float m1 = x_ml[r], l1 = x_ml[kBM + r];
          const float mm = fmaxf(m, m1);
          a0 = ex2_approx(m - mm);
          a1 = ex2_approx(m1 - mm);
          l = a0 * l + a1 * l1;
          m = mm;
        }
      }
      tc_fence_after();
      const int n = cnt_of(p, s_cnt, b);
      const int i = (2 * pair + qtile) * kBM + r;
      const bool store = i < n;
      const bool partial = wslot >= 0;
      const float inv = partial ? 1.0f : 1.0f / l;
      const float w0 = a0 * inv, w1 = a1 * inv;
      const int64_t slot = (int64_t)wslot * 2 + qtile;  // workspace tile slot (split items)
      __nv_bfloat16* orow =
          p.o + ((int64_t)b * p.M_max + i) * ((int64_t)p.H * kHD) + (int64_t)h * kHD;
      float* prow = p.ws_o + (slot * kBM + r) * kHD;
#pragma unroll 1
      for (int c = 0; c < (idle ? 0 : kHD / 32); ++c) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tO + c * 32, ov);
        if (merge) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t o1[16];
            tmem_ld_32x32b_x16(tO1 + c * 32 + hf * 16, o1);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 16; ++q)
              ov[hf * 16 + q] = __float_as_uint(
                  fmaf(__uint_as_float(ov[hf * 16 + q]), w0, __uint_as_float(o1[q]) * w1));
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 32; ++q) ov[q] = __float_as_uint(__uint_as_float(ov[q]) * w0);
        }
        if (store && partial) {
          float4* dst = reinterpret_cast<float4*>(prow + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(ov[q * 4 + 0]), __uint_as_float(ov[q * 4 + 1]),
                                 __uint_as_float(ov[q * 4 + 2]), __uint_as_float(ov[q * 4 + 3]));
        } else if (store) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(ov[q * 8 + 0]), __uint_as_float(ov[q * 8 + 1]));
            w.y = pack_bf16(__uint_as_float(ov[q * 8 + 2]), __uint_as_float(ov[q * 8 + 3]));
            w.z = pack_bf16(__uint_as_float(ov[q * 8 + 4]), __uint_as_float(ov[q * 8 + 5]));
            w.w = pack_bf16(__uint_as_float(ov[q * 8 + 6]), __uint_as_float(ov[q * 8 + 7]));
            dst[q] = w;
          }
        }
      }
      // O is read: the next item's first P V may overwrite it (both slots'
      // O after a merged one-tile item).
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&o_free[x]);
        if (merge) mbar_arrive(&o_free[1]);
      }
      if (store) {
        if (partial) {
          p.ws_ml[(slot * kBM + r) * 2 + 0] = m;
          p.ws_ml[(slot * kBM + r) * 2 + 1] = l;
        } else if (p.lse != nullptr) {
          p.lse[((int64_t)b * p.H + h) * p.M_max + i] = (m + log2f(l)) * 0.69314718055994531f;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpTma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort) report(p.dev_status, DLLM_ERR_TIMEOUT);
}

// Combines the key-range splits of each active row of the split pairs:
// O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, lse = (M + log2 l) ln 2.
// One warp per (split pair, tile, row), each lane four of the 128 dims;
// does nothing when the plan split no pair.
__global__ void __launch_bounds__(256)
attn_split_merge_kernel(FwdParams p, int n_ctas) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  __shared__ int s_cnt[kPlanMaxB];
  stage_counts(p, s_cnt);
  __syncthreads();
  const FwdPlan plan = make_plan(p, s_cnt, n_ctas);
  if (plan.nsplit <= 1) return;
  const int lane = threadIdx.x & 31;
  const int64_t total = (int64_t)(plan.total_qp - plan.n_full) * 2 * kBM;
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total;
       w += (int64_t)gridDim.x * (blockDim.x >> 5)) {
    const int sp = (int)(w / (2 * kBM));  // split pair
    const int x = (int)((w / kBM) & 1);   // tile of the pair
    const int r = (int)(w % kBM);         // row of the tile
    int b, h, pair, nq;
    decode_pair(p, s_cnt, plan.n_full + sp, &b, &h, &pair, &nq);
    if (x >= nq) continue;
    const int i = (2 * pair + x) * kBM + r;
    if (i >= cnt_of(p, s_cnt, b)) continue;
    // all loads of the row's slices are issued before any is used
    constexpr int kU = 4;
    float M = -INFINITY, l = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < plan.nsplit; s0 += kU) {
      float2 ml[kU];
      float4 o4[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (s0 + u < plan.nsplit) {
          const int64_t slot = ((int64_t)sp * plan.nsplit + s0 + u) * 2 + x;
          ml[u] = __ldca(reinterpret_cast<const float2*>(p.ws_ml + (slot * kBM + r) * 2));
          o4[u] = __ldca(reinterpret_cast<const float4*>(p.ws_o + (slot * kBM + r) * kHD) + lane);
        } else {
          ml[u] = make_float2(-INFINITY, 0.f);
          o4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float Mn = M;
#pragma unroll
      for (int u = 0; u < kU; ++u) Mn = fmaxf(Mn, ml[u].x);
      const float c = ex2_approx(M - Mn);  // rescale what was accumulated so far
      l *= c;
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] *= c;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const float wgt = ex2_approx(ml[u].x - Mn);
        l = fmaf(wgt, ml[u].y, l);
        acc[0] = fmaf(wgt, o4[u].x, acc[0]);
        acc[1] = fmaf(wgt, o4[u].y, acc[1]);
        acc[2] = fmaf(wgt, o4[u].z, acc[2]);
        acc[3] = fmaf(wgt, o4[u].w, acc[3]);
      }
      M = Mn;
    }
    const float inv = 1.0f / l;
    __nv_bfloat16* orow =
        p.o + ((int64_t)b * p.M_max + i) * ((int64_t)p.H * kHD) + (int64_t)h * kHD;
    uint2 w2;
    w2.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    w2.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    reinterpret_cast<uint2*>(orow)[lane] = w2;
    if (lane == 0 && p.lse != nullptr)
      p.lse[((int64_t)b * p.H + h) * p.M_max + i] = (M + log2f(l)) * 0.69314718055994531f;
  }
}

// Column sums, the second normalised pass.  One CTA per (NK consecutive key
// tiles of 128 keys, head, batch row); NK in {1, 2, 4} is chosen on the host
// so that the grid still covers the SMs.  Warps 0..4NK-1 form NK softmax
// warpgroups (key tile X = warp / 4; thread = one key, its TMEM lane), warp
// 4NK is the TMA producer (the NK key tiles once, then the query tiles of
// 128 active rows into a 2-stage ring), warp 4NK+1 issues the MMAs:
// S_X^T = K_X Q^T for every key tile X of the CTA into its own 128 TMEM
// columns, so one query tile feeds NK key tiles and NK warps per scheduler
// hide each other's latency.  A thread reads its S row in chunks of 32
// queries, releases S_X after the last chunk is read, and adds
// 2^(s * scale * log2 e - lse * log2 e) over the active rows; -lse (log2
// units, -inf for padded rows) sits in a warp-private shared buffer,
// prefetched one query tile ahead.  Each key has one owner thread: no
// atomics, run-to-run identical.
template <int NK>
__global__ void __launch_bounds__((4 * NK + 2) * 32, 1)
attn_colsum_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      ColsumParams p) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  constexpr int kSoftWarps = 4 * NK;
  constexpr uint32_t kTmCols = NK == 1 ? 128 : NK * 128;
  const int kg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  int n = __ldca(p.count + b);
  n = n < 0 ? 0 : (n > p.M_max ? p.M_max : n);
  const int nqt = (n + kBM - 1) / kBM;
  if (nqt < p.min_qt) return;  // the persistent kernel covers this batch row
  const int nkt = (p.L + kBN - 1) / kBN;
  const int nk = min(NK, nkt - kg * NK);  // key tiles of this CTA
  const int key_base = kg * NK * kBN;
  float* out = p.colsum + ((int64_t)b * p.H + h) * p.L;
  if (nqt == 0) {
    for (int j = threadIdx.x; j < NK * kBN; j += blockDim.x)
      if (key_base + j < p.L) out[key_base + j] = 0.f;
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  constexpr uint32_t oQ = NK * kTile;                       // Q ring
  constexpr uint32_t oL = oQ + kStages * kTile;             // warp-private -lse buffers
  constexpr uint32_t oBar = oL + kSoftWarps * 2 * kBM * 4;
  float* lse_w = reinterpret_cast<float*>(gbase + oL);      // [warp][2][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + oBar);
  uint64_t* k_full = bars + 0;
  uint64_t* q_full = bars + 1;             // [kStages]
  uint64_t* q_empty = bars + 1 + kStages;  // [kStages]
  uint64_t* s_full = bars + 1 + 2 * kStages;        // [NK]
  uint64_t* s_free = bars + 1 + 2 * kStages + NK;   // [NK]
  uint64_t* mma_done = bars + 1 + 2 * kStages + 2 * NK;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* abort_flag = reinterpret_cast<int*>(mma_done + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kWarpT = kSoftWarps, kWarpM = kSoftWarps + 1;
  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int x = 0; x < NK; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&s_free[x], 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpT) tmem_alloc(tmem_slot, kTmCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort = abort_flag;

  if (warp == kWarpT) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      const uint64_t pol_k = l2_policy_evict_first();  // the keys' last read of the step
      mbar_expect_tx(k_full, (uint32_t)nk * kTile);
      for (int x = 0; x < nk; ++x) {
        const int key0 = key_base + x * kBN;
        tma_load_4d_hint(gbase + x * kTile, &tk, k_full, 0, h, key0, b, pol_k);
        tma_load_4d_hint(gbase + x * kTile + kBox, &tk, k_full, 64, h, key0, b, pol_k);
      }
      int issued = 0;
      for (int it = 0; it < nqt; ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mbar_wait(&q_empty[s], ((it / kStages) - 1) & 1, abort)) break;
        uint8_t* qdst = gbase + oQ + s * kTile;
        mbar_expect_tx(&q_full[s], kTile);
        tma_load_4d(qdst, &tq, &q_full[s], 0, h, it * kBM, b);
        tma_load_4d(qdst + kBox, &tq, &q_full[s], 64, h, it * kBM, b);
        issued = it + 1;
      }
      int none = 0;
      mbar_wait(k_full, 0, &none);
      for (int it = issued - kStages < 0 ? 0 : issued - kStages; it < issued; ++it)
        mbar_wait(&q_full[it % kStages], (it / kStages) & 1, &none);
      if (none) report(p.dev_status, DLLM_ERR_TIMEOUT);
    }
  } else if (warp == kWarpM) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id = idesc_bf16_f32(kBN, kBM, false, false);
      bool ok = mbar_wait(k_full, 0, abort);
      for (int it = 0; ok && it < nqt; ++it) {
        const int s = it % kStages;
        if (!mbar_wait(&q_full[s], (it / kStages) & 1, abort)) break;
        const uint32_t sQ = base + oQ + s * kTile;
        for (int x = 0; x < nk; ++x) {
          if (it > 0 && !mbar_wait(&s_free[x], (it - 1) & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sK = base + x * kTile;
#pragma unroll
          for (int kk = 0; kk < kHD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
            mma_bf16_ss(tmem + x * kBN, smem_desc_sw128(sK + off, 16, 1024),
                        smem_desc_sw128(sQ + off, 16, 1024), id, kk > 0);
          }
          mma_commit(&s_full[x]);
        }
        if (ok) mma_commit(&q_empty[s]);
      }
      mma_commit(mma_done);
      int none = 0;
      mbar_wait(mma_done, 0, &none);
      if (none) report(p.dev_status, DLLM_ERR_TIMEOUT);
    }
  } else if (warp / 4 < nk) {
    // ------------------------------------------------------------ softmax warps
    const int x = warp >> 2;
    const int quarter = warp & 3;
    const int j = quarter * 32 + lane;  // key of this thread within its tile
    const uint32_t tS = tmem + ((uint32_t)(quarter * 32) << 16) + x * kBN;
    const float* lse_g = p.lse + ((int64_t)b * p.H + h) * p.M_max;
    float* lbuf = lse_w + warp * 2 * kBM;
    const float sl2 = p.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
    // -lse (log2 units) of query rows lane + 32 q of tile it, -inf past the count
    auto load_lse = [&](int it, float (&v)[4]) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = it * kBM + q * 32 + lane;
        v[q] = (it < nqt && i < n) ? -__ldca(lse_g + i) * kLog2e : -INFINITY;
      }
    };
    float nl[4];
    load_lse(0, nl);
    bool ok = true;
    for (int it = 0; ok && it < nqt; ++it) {
      float* lb = lbuf + (it & 1) * kBM;
#pragma unroll
      for (int q = 0; q < 4; ++q) lb[q * 32 + lane] = nl[q];
      __syncwarp();
      load_lse(it + 1, nl);  // the next tile's values, while this tile is worked on
      if (!warp_wait(&s_full[x], it & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the S row in 8 chunks of 16 queries, two register buffers: the next
      // chunk's scores load while this one is summed
      auto add16 = [&](const uint32_t(&rw)[16], int c16) {
        const float4* nl4 = reinterpret_cast<const float4*>(lb + c16 * 16);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 L4 = nl4[q4];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int q = q4 * 4 + hh * 2;
            const float2 a = __ffma2_rn(
                make_float2(__uint_as_float(rw[q]), __uint_as_float(rw[q + 1])), sl2x2,
                hh ? make_float2(L4.z, L4.w) : make_float2(L4.x, L4.y));
            float2 e;
            if ((((c16 * 16 + q) >> 1) & 7) >= 8 - kColsumGroupPoly) {
              e = exp2_poly2(a);
            } else {
              e.x = ex2_approx(a.x);
              e.y = ex2_approx(a.y);
            }
            if (hh)
              acc1 = __fadd2_rn(acc1, e);
            else
              acc0 = __fadd2_rn(acc0, e);
          }
        }
      };
      uint32_t ra[16], rb[16];
      tmem_ld_32x32b_x16(tS, ra);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < kBM / 16; c += 2) {
        tmem_ld_32x32b_x16(tS + (c + 1) * 16, rb);
        add16(ra, c);
        tmem_ld_wait();
        if (c + 2 < kBM / 16) {
          tmem_ld_32x32b_x16(tS + (c + 2) * 16, ra);
        } else {  // S_X is read: the next query tile may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_free[x]);
        }
        add16(rb, c + 1);
        if (c + 2 < kBM / 16) tmem_ld_wait();
      }
      __syncwarp();  // lb is rewritten two tiles later
    }
    const int key = key_base + x * kBN + j;
    if (ok && key < p.L) out[key] = (acc0.x + acc0.y) + (acc1.x + acc1.y);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpT) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmCols);
  }
  if (threadIdx.x == 0 && *abort) report(p.dev_status, DLLM_ERR_TIMEOUT);
}

// Column sums of batch rows with at most two query tiles (the small active
// sets of most steps), persistent: one CTA per SM takes a contiguous range of
// (batch row, head, key tile) items.  Warp 8 loads the query tiles of a head
// once (they stay resident while its key tiles pass) and streams the key
// tiles through a four-stage ring; warp 9 issues S^T = K Q^T for each query
// tile of the item into the TMEM of softmax warpgroup g = item % 2, so one
// warpgroup adds up the exponentials of one key tile while the tensor cores
// and the other warpgroup work on the next.  Each softmax thread owns one
// key: it adds 2^(s * scale * log2 e - lse * log2 e) over the active query
// rows (chunks of 32 queries past the count are skipped; -lse sits in a
// warp-private shared buffer per head) and writes the key's column sum.  Rows
// with no active query get zeros.  Each key has one owner thread: no atomics,
// run-to-run identical.
//
// When every batch row of the CTA's range has at most one query tile (S^T
// then takes 128 TMEM columns), each warpgroup gets two S buffers, so the
// product of its next item is ready when it finishes the current one, and the
// query tiles of consecutive heads go to alternate Q slots, so the next
// head's query tile loads while the current head's last products run.
constexpr int kCsThreads = 320;  // warps 0-7 softmax (two groups), 8 TMA, 9 MMA
constexpr int kCsKStages = 4;
constexpr uint32_t kCsQ = 0;                                   // kCsMaxQt query tiles
constexpr uint32_t kCsK = kCsMaxQt * kTile;                    // + s * kTile
constexpr uint32_t kCsL = kCsK + kCsKStages * kTile;           // [8 warps][256] -lse log2 e
constexpr uint32_t kCsBar = kCsL + 8 * kCsMaxQt * kBM * 4;
constexpr uint32_t kCsSmem = kCsBar + 256 + 1024;

__global__ void __launch_bounds__(kCsThreads, 1)
attn_colsum_stream_kernel(const __grid_constant__ CUtensorMap tq,
                          const __grid_constant__ CUtensorMap tk, ColsumParams p, int B) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kCsBar);
  uint64_t* q_full = bars + 0;   // [2] Q slots
  uint64_t* q_empty = bars + 2;  // [2]
  uint64_t* k_full = bars + 4;                // [kCsKStages]
  uint64_t* k_empty = bars + 4 + kCsKStages;  // [kCsKStages]
  uint64_t* s_full = bars + 4 + 2 * kCsKStages;  // [group * 2 + buffer]
  uint64_t* s_free = bars + 8 + 2 * kCsKStages;  // [group * 2 + buffer] (4 warps each)
  uint64_t* mma_done = bars + 12 + 2 * kCsKStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13 + 2 * kCsKStages);
  int* abort_flag = reinterpret_cast<int*>(bars + 14 + 2 * kCsKStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < kCsKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) tmem_alloc(tmem_slot, 512);
  __shared__ int s_nqt[kPlanMaxB];      // query tiles of each batch row; -1: not handled here
  __shared__ int s_n[kPlanMaxB];        // active rows of each batch row (clamped)
  __shared__ int s_first[kPlanMaxB + 1];  // first item of each batch row
  const int nkt = (p.L + kBN - 1) / kBN;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      int n = __ldca(p.count + b);
      n = n < 0 ? 0 : (n > p.M_max ? p.M_max : n);
      const int nqt = (n + kBM - 1) / kBM;
      s_n[b] = n;
      s_first[b] = acc;
      s_nqt[b] = nqt <= kCsMaxQt ? nqt : -1;
      if (nqt <= kCsMaxQt) acc += p.H * nkt;
    }
    s_first[B] = acc;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort = abort_flag;
  const int N = s_first[B];
  const int i0 = (int)((long long)blockIdx.x * N / gridDim.x);
  const int i1 = (int)((long long)(blockIdx.x + 1) * N / gridDim.x);
  if (i0 >= i1) {  // no work: give the tensor memory back
    if (warp == 8) tmem_dealloc(tmem, 512);
    return;
  }
  // double buffering of S and Q: every batch row in [i0, i1) has <= 1 query tile
  bool dbl = true;
  for (int b = 0; b < B; ++b)
    if (s_nqt[b] > 1 && s_first[b] < i1 && s_first[b + 1] > i0) dbl = false;
  // item i -> (b, h, kt).  The key tiles of a head are taken last first:
  // the forward pass that usually runs just before streams every head's key
  // tiles first to last, so its last tiles are the ones still in L2.
  auto decode = [&](int i, int* b, int* h, int* kt) {
    int bb = 0;
    while (s_nqt[bb] < 0 || i >= s_first[bb + 1]) ++bb;
    const int r = i - s_first[bb];
    *b = bb;
    *h = r / nkt;
    *kt = nkt - 1 - (r - *h * nkt);
  };
  // the n-th item with query tiles of a warpgroup uses S buffer sbuf(n), for
  // the suse(n)-th time; the sq-th head uses Q slot qslot(sq) for the
  // quse(sq)-th time
  auto sbuf = [&](int n) { return dbl ? (n & 1) : 0; };
  auto suse = [&](int n) { return dbl ? (n >> 1) : n; };
  auto qslot = [&](int sq) { return dbl ? (sq & 1) : 0; };
  auto quse = [&](int sq) { return dbl ? (sq >> 1) : sq; };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_k = l2_policy_evict_first();  // the keys' last read of the step
      int kc = 0, sq = 0, cur = -1;
      for (int i = i0; i < i1; ++i) {
        int b, h, kt;
        decode(i, &b, &h, &kt);
        const int nqt = s_nqt[b];
        if (nqt == 0) continue;
        if (b * p.H + h != cur) {  // a new head: its query tiles, once
          const int qs = qslot(sq), qu = quse(sq);
          if (qu > 0 && !mbar_wait(&q_empty[qs], (qu - 1) & 1, abort)) break;
          mbar_expect_tx(&q_full[qs], (uint32_t)nqt * kTile);
          for (int qt = 0; qt < nqt; ++qt) {
            uint8_t* qdst = gbase + kCsQ + (qs + qt) * kTile;
            tma_load_4d(qdst, &tq, &q_full[qs], 0, h, qt * kBM, b);
            tma_load_4d(qdst + kBox, &tq, &q_full[qs], 64, h, qt * kBM, b);
          }
          cur = b * p.H + h;
          ++sq;
        }
        const int s = kc % kCsKStages;
        if (kc >= kCsKStages && !mbar_wait(&k_empty[s], ((kc / kCsKStages) - 1) & 1, abort))
          break;
        mbar_expect_tx(&k_full[s], kTile);
        tma_load_4d_hint(gbase + kCsK + s * kTile, &tk, &k_full[s], 0, h, kt * kBN, b, pol_k);
        tma_load_4d_hint(gbase + kCsK + s * kTile + kBox, &tk, &k_full[s], 64, h, kt * kBN, b,
                         pol_k);
        ++kc;
      }
      // Drain: the query tiles of the last head of each slot (earlier ones
      // were consumed before their slot was reused) and the last key tiles.
      int none = 0;
      for (int s = sq - (dbl ? 2 : 1) < 0 ? 0 : sq - (dbl ? 2 : 1); s < sq; ++s)
        mbar_wait(&q_full[qslot(s)], quse(s) & 1, &none);
      for (int k = kc - kCsKStages < 0 ? 0 : kc - kCsKStages; k < kc; ++k)
        mbar_wait(&k_full[k % kCsKStages], (k / kCsKStages) & 1, &none);
      if (none) report(p.dev_status, DLLM_ERR_TIMEOUT);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id = idesc_bf16_f32(kBN, kBM, false, false);
      int kc = 0, sq = 0, cur = -1, cq = 0;
      int ng[2] = {0, 0};  // items with query tiles per softmax group
      bool ok = true;
      for (int i = i0; ok && i < i1; ++i) {
        int b, h, kt;
        decode(i, &b, &h, &kt);
        const int nqt = s_nqt[b];
        if (nqt == 0) continue;
        const int g = (i - i0) & 1;
        if (b * p.H + h != cur) {
          // every product with the previous head's query tiles is issued
          if (sq > 0) mma_commit(&q_empty[qslot(sq - 1)]);
          if (!mbar_wait(&q_full[qslot(sq)], quse(sq) & 1, abort)) break;
          cq = qslot(sq);
          cur = b * p.H + h;
          ++sq;
        }
        const int s = kc % kCsKStages;
        if (!mbar_wait(&k_full[s], (kc / kCsKStages) & 1, abort)) break;
        const int sb = sbuf(ng[g]), su = suse(ng[g]);
        if (su > 0 && !mbar_wait(&s_free[g * 2 + sb], (su - 1) & 1, abort)) break;
        tc_fence_after();
        const uint32_t sK = base + kCsK + s * kTile;
        for (int qt = 0; qt < nqt; ++qt) {
          const uint32_t sQ = base + kCsQ + (cq + qt) * kTile;
#pragma unroll
          for (int kk = 0; kk < kHD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
            mma_bf16_ss(tmem + g * 256 + sb * 128 + qt * kBM, smem_desc_sw128(sK + off, 16, 1024),
                        smem_desc_sw128(sQ + off, 16, 1024), id, kk > 0);
          }
        }
        mma_commit(&s_full[g * 2 + sb]);
        mma_commit(&k_empty[s]);
        ++kc;
        ++ng[g];
      }
      mma_commit(mma_done);
      int none = 0;
      mbar_wait(mma_done, 0, &none);
      if (none) report(p.dev_status, DLLM_ERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int g = warp >> 2;
    const int quarter = warp & 3;
    const int j = quarter * 32 + lane;  // key of this thread within the tile
    const uint32_t tS0 = tmem + ((uint32_t)(quarter * 32) << 16) + g * 256;
    float* lb = reinterpret_cast<float*>(gbase + kCsL) + warp * (kCsMaxQt * kBM);
    const float sl2 = p.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    int ng = 0, cur = -1, n = 0;
    bool ok = true;
    for (int i = i0 + g; ok && i < i1; i += 2) {
      int b, h, kt;
      decode(i, &b, &h, &kt);
      const int nqt = s_nqt[b];
      const int key = kt * kBN + j;
      float* out = p.colsum + ((int64_t)b * p.H + h) * p.L;
      if (nqt == 0) {
        if (key < p.L) out[key] = 0.f;
        continue;
      }
      if (b * p.H + h != cur) {  // -lse (log2 units) of the head's query rows, -inf past the count
        cur = b * p.H + h;
        n = s_n[b];
        const float* lse_g = p.lse + ((int64_t)b * p.H + h) * p.M_max;
        constexpr int kPer = kCsMaxQt * kBM / 32;
        float v[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {  // all loads first, then the stores
          const int q = lane + 32 * u;
          v[u] = q < n ? __ldca(lse_g + q) : INFINITY;
        }
        __syncwarp();
#pragma unroll
        for (int u = 0; u < kPer; ++u) lb[lane + 32 * u] = -v[u] * kLog2e;
        __syncwarp();
      }
      const int sb = sbuf(ng), su = suse(ng);
      if (!warp_wait(&s_full[g * 2 + sb], su & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tS0 + sb * 128;
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      const int nch = (n + 31) / 32;  // chunks of 32 queries holding an active row
      auto add_chunk = [&](const uint32_t(&rw)[32], int c) {
        const float4* nl4 = reinterpret_cast<const float4*>(lb + c * 32);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 L4 = nl4[q4];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int q = q4 * 4 + hh * 2;
            const float2 a = __ffma2_rn(make_float2(__uint_as_float(rw[q]), __uint_as_float(rw[q + 1])),
                                        sl2x2, hh ? make_float2(L4.z, L4.w) : make_float2(L4.x, L4.y));
            float2 e;
            if (((q >> 1) & 7) >= 8 - kColsumPoly) {
              e = exp2_poly2(a);
            } else {
              e.x = ex2_approx(a.x);
              e.y = ex2_approx(a.y);
            }
            if (hh)
              acc1 = __fadd2_rn(acc1, e);
            else
              acc0 = __fadd2_rn(acc0, e);
          }
        }
      };
      // two register buffers: the next chunk's scores load while one is summed
      uint32_t ra[32], rb[32];
      tmem_ld_32x32b_x32(tS, ra);
      tmem_ld_wait();
      for (int c = 0; c < nch; c += 2) {
        if (c + 1 < nch) tmem_ld_32x32b_x32(tS + (c + 1) * 32, rb);
        add_chunk(ra, c);
        tmem_ld_wait();
        if (c + 1 < nch) {
          if (c + 2 < nch) tmem_ld_32x32b_x32(tS + (c + 2) * 32, ra);
          add_chunk(rb, c + 1);
          tmem_ld_wait();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[g * 2 + sb]);  // this S buffer may be overwritten
      ++ng;
      if (key < p.L) out[key] = (acc0.x + acc0.y) + (acc1.x + acc1.y);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort) report(p.dev_status, DLLM_ERR_TIMEOUT);
}

template <int NK>
constexpr uint32_t colsum_smem_bytes() {
  return NK * kTile + kStages * kTile + 4 * NK * 2 * kBM * 4 + 256 + 1024;
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

size_t attention_tc_workspace_bytes(int n_ctas) {
  // at most 2 x n_ctas split items of two 128-row tiles: unnormalised O (128
  // floats) + (max, sum) per row
  return (size_t)2 * n_ctas * 2 * kBM * (kHD + 2) * sizeof(float);
}

cudaError_t launch_attention_tc(const void* q, const void* k, const void* v, int B, int L, int H,
                                int M_max, const int32_t* count, float scale, void* o, float* lse,
                                float* colsum, void* ws, size_t ws_bytes, int32_t* dev_status,
                                cudaStream_t stream) {
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(attn_fwd_tc_kernel),
                                    (int)kFwdSmem);
  if (e != cudaSuccess) return e;
  CUtensorMap tq, tk, tv;
  if (!make_rows_map(&tq, q, B, M_max, H) || !make_rows_map(&tk, k, B, L, H) ||
      !make_rows_map(&tv, v, B, L, H))
    return cudaErrorInvalidValue;
  const int n_ctas = num_sms();
  const size_t need = attention_tc_workspace_bytes(n_ctas);
  // Splitting the key range costs the merge launch (about 4 us with its
  // start-up): below kMinSplitTiles key tiles a CTA's whole range takes
  // less than that (L 1024, 32 heads: 14.7 us unsplit against 16.4 us split
  // and merged; L 2048: 23.4 against 19.3 us).
  const int nkt = (L + kBN - 1) / kBN;
  const bool can_split = ws != nullptr && ws_bytes >= need &&
                         reinterpret_cast<uintptr_t>(ws) % 16 == 0 && nkt >= kMinSplitTiles;
  FwdParams fp;
  fp.count = count;
  fp.o = static_cast<__nv_bfloat16*>(o);
  fp.lse = lse;
  fp.ws_o = can_split ? static_cast<float*>(ws) : nullptr;
  fp.ws_ml = can_split ? static_cast<float*>(ws) + (size_t)2 * n_ctas * 2 * kBM * kHD : nullptr;
  fp.B = B;
  fp.L = L;
  fp.H = H;
  fp.M_max = M_max;
  fp.max_split_items = can_split ? 2 * n_ctas : 0;
  fp.scale_log2 = scale * kLog2e;
  fp.dev_status = dev_status;
  fp.wait_limit = wait_limit();
  launch_pdl(attn_fwd_tc_kernel, n_ctas, kFwdThreads, kFwdSmem, stream, tq, tk, tv, fp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (can_split) {
    // one warp per (split pair, tile, row): up to 64 warps per SM
    launch_pdl(attn_split_merge_kernel, 8 * n_ctas, 256, 0, stream, fp, n_ctas);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (colsum == nullptr) return cudaSuccess;
  return launch_colsum_tc(q, k, B, L, H, M_max, count, scale, lse, colsum, dev_status, stream);
}

cudaError_t launch_colsum_tc(const void* q, const void* k, int B, int L, int H, int M_max,
                             const int32_t* count, float scale, const float* lse, float* colsum,
                             int32_t* dev_status, cudaStream_t stream) {
  CUtensorMap tq, tk;
  if (!make_rows_map(&tq, q, B, M_max, H) || !make_rows_map(&tk, k, B, L, H))
    return cudaErrorInvalidValue;
  ColsumParams cp{count, lse, colsum, L, H, M_max, scale * kLog2e, dev_status, 0};
  const int nkt = (L + kBN - 1) / kBN;
  const int64_t bh = (int64_t)B * H;
  const int sms = num_sms();
  cudaError_t e;
  if (B <= kPlanMaxB && bh * nkt >= 4 * (int64_t)sms) {
    // batch rows with at most kCsMaxQt query tiles: the persistent kernel
    // (when there are at least four key tiles per SM to amortise its
    // set-up); the key-tile-group kernel below then takes only the larger
    // ones
    e = ensure_smem_limit(reinterpret_cast<const void*>(attn_colsum_stream_kernel), (int)kCsSmem);
    if (e != cudaSuccess) return e;
    launch_pdl(attn_colsum_stream_kernel, sms, kCsThreads, kCsSmem, stream, tq, tk, cp, B);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (M_max <= kCsMaxQt * kBM) return cudaSuccess;  // no row can have more query tiles
    cp.min_qt = kCsMaxQt + 1;
  }
  // Key tiles per CTA: 4 (one query tile feeds four key tiles, four warps
  // per scheduler) while that still leaves two CTAs per SM, else fewer.
  if (bh * ((nkt + 3) / 4) >= 2 * sms) {
    e = ensure_smem_limit(reinterpret_cast<const void*>(attn_colsum_tc_kernel<4>),
                          (int)colsum_smem_bytes<4>());
    if (e != cudaSuccess) return e;
    dim3 grid((nkt + 3) / 4, H, B);
    launch_pdl(attn_colsum_tc_kernel<4>, grid, 18 * 32, colsum_smem_bytes<4>(), stream, tq, tk, cp);
  } else if (bh * ((nkt + 1) / 2) >= sms) {
    e = ensure_smem_limit(reinterpret_cast<const void*>(attn_colsum_tc_kernel<2>),
                          (int)colsum_smem_bytes<2>());
    if (e != cudaSuccess) return e;
    dim3 grid((nkt + 1) / 2, H, B);
    launch_pdl(attn_colsum_tc_kernel<2>, grid, 10 * 32, colsum_smem_bytes<2>(), stream, tq, tk, cp);
  } else {
    e = ensure_smem_limit(reinterpret_cast<const void*>(attn_colsum_tc_kernel<1>),
                          (int)colsum_smem_bytes<1>());
    if (e != cudaSuccess) return e;
    dim3 grid(nkt, H, B);
    launch_pdl(attn_colsum_tc_kernel<1>, grid, 6 * 32, colsum_smem_bytes<1>(), stream, tq, tk, cp);
  }
  return cudaGetLastError();
}

}  // namespace dllm
