// Approximate attention update of the stable rows on the tensor cores (bf16,
// head dim 128).
//
// DyLLM ("DyLLM: Efficient Diffusion LLM Inference via Saliency-based Token
// Selection and Partial Attention"), technical summary, Methodology 2
// (non-salient path): a stable row keeps its attention weights and its output
// moves by the change of the salient tokens' values weighted by them, cost
// O(N |A_t|).  For the stable rows Q_S, the previous keys K_A and values V_A
// of the salient positions and their fresh values V'_A:
//   S = Q_S K_A^T,  P = 2^(S scale log2 e - lse log2 e),  O_S += P V'_A - P V_A.
// Both products are dense contractions, so they run on tcgen05: S into one
// 128-column TMEM tile, P and -P written back over it as bf16 pairs, and the
// two P V products accumulated into a second TMEM tile (the value change is
// never rounded: the fresh and the previous values each enter exactly, with
// -P for the previous ones).
//
// approx_update_tc_kernel  one CTA of 128 threads per (128 stable rows, head,
//   batch row), at most two per SM (256 TMEM columns each).
//   The gathered rows (stable queries, salient keys and values) are copied
//   with cp.async straight into the 128-byte-swizzled operand layout of the
//   MMA; two 32 KB buffers hold Q and K_A for S, then V'_A and V_A (loaded
//   while the softmax of S runs).  Each thread owns one stable row: its
//   probabilities, then its output row, read, updated in float32 and
//   rounded once.  More than 128 salient columns are taken 128 at a time.
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace dllm {
namespace {

using namespace sm100;

constexpr int kTuThreads = 128;
constexpr int kTuRows = 128;     // stable rows per CTA
constexpr int kTuCols = 128;     // salient columns per pass
constexpr int kTuD = 128;        // head dim
constexpr uint32_t kTuBox = 16384;             // 128 rows x 64 dims, swizzled
constexpr uint32_t kTuTile = 2 * kTuBox;        // 128 rows x 128 dims
// two 32 KB operand buffers, barriers and alignment slack, padded so that at
// most two CTAs share an SM (their 2 x 256 TMEM columns then always fit)
constexpr uint32_t kTuSmem = 100 * 1024;
static_assert(2 * kTuTile + 256 + 1024 <= kTuSmem, "shared-memory map");
constexpr uint32_t kTmS = 0;     // S, then P (columns 0-63) and -P (64-127)
constexpr uint32_t kTmO = 128;   // the output change

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void st_shared_zero16(uint32_t smem) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(smem), "r"(0) : "memory");
}

// Row r of a 128 x 128 bf16 tile at `tile` (two 64-dim boxes, 128-byte
// swizzle: 16-byte chunk c of a 128-byte row r sits at chunk c ^ (r % 8)),
// from the 256-byte row at `src`, or zeros when src is null.
__device__ __forceinline__ void load_row(uint32_t tile, int r, const __nv_bfloat16* src) {
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint32_t dst = tile + (uint32_t)(c >> 3) * kTuBox + (uint32_t)r * 128u +
                         ((uint32_t)((c & 7) ^ (r & 7)) << 4);
    if (src != nullptr)
      cp_async16(dst, src + c * 8);
    else
      st_shared_zero16(dst);
  }
}

__global__ void __launch_bounds__(kTuThreads)
approx_update_tc_kernel(const __nv_bfloat16* q, const float* lse, const __nv_bfloat16* k,
                        const __nv_bfloat16* v, const __nv_bfloat16* v_new, const int32_t* idx,
                        const int32_t* count, const int32_t* stable_idx,
                        const int32_t* stable_count, __nv_bfloat16* o, int L, int H, int M_max,
                        int N_max, float scale_log2e, int32_t* dev_status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  const int b = blockIdx.z, h = blockIdx.y, r0 = blockIdx.x * kTuRows;
  const int t = threadIdx.x, warp = t >> 5;
  int ns = __ldca(stable_count + b);
  int na = __ldca(count + b);
  if (ns < 0 || ns > N_max || na < 0 || na > M_max) {
    if (t == 0 && blockIdx.x == 0 && h == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
    ns = ns < 0 ? 0 : (ns > N_max ? N_max : ns);
    na = na < 0 ? 0 : (na > M_max ? M_max : na);
  }
  if (r0 >= ns || na == 0) return;  // uniform over the CTA

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  const uint32_t X = base, Y = base + kTuTile;  // Q, then V'_A | K_A, then V_A
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + 2 * kTuTile);
  uint64_t* s_full = bars + 0;
  uint64_t* o_done = bars + 1;
  uint64_t* drained = bars + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3);
  int* abort_flag = reinterpret_cast<int*>(bars + 4);
  if (t == 0) {
    mbar_init(s_full, 1);
    mbar_init(o_done, 1);
    mbar_init(drained, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort = abort_flag;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tmem + lane_base + kTmS, tO = tmem + lane_base + kTmO;

  // this thread's stable row
  int pos = -1;
  if (r0 + t < ns) {
    pos = __ldca(stable_idx + (int64_t)b * N_max + r0 + t);
    if (pos < 0 || pos >= L) {
      if (h == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
      pos = -1;
    }
  }
  const int64_t rs = (int64_t)H * kTuD;  // elements between positions
  const __nv_bfloat16* qrow = pos >= 0 ? q + ((int64_t)b * L + pos) * rs + (int64_t)h * kTuD : nullptr;
  const float nl = pos >= 0 ? -__ldca(lse + ((int64_t)b * H + h) * L + pos) * kLog2e : 0.f;
  const uint32_t id_qk = idesc_bf16_f32(kTuRows, kTuCols, false, false);
  const uint32_t id_pv = idesc_bf16_f32(kTuRows, kTuD, false, true);

  bool ok = true;
  int phase = 0;
  for (int a0 = 0; ok && a0 < na; a0 += kTuCols, phase ^= 1) {
    // this thread's salient column a0 + t: its position, previous key and values
    int apos = -1;
    if (a0 + t < na) {
      apos = __ldca(idx + (int64_t)b * M_max + a0 + t);
      if (apos < 0 || apos >= L) {
        if (h == 0 && blockIdx.x == 0) report(dev_status, DLLM_ERR_DEVICE_CHECK);
        apos = -1;
      }
    }
    const int64_t aoff = ((int64_t)b * L + apos) * rs + (int64_t)h * kTuD;
    // 1. Q_S and K_A, then S = Q_S K_A^T
    load_row(X, t, qrow);
    load_row(Y, t, apos >= 0 ? k + aoff : nullptr);
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTuD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kTuBox + (kk & 3) * 32;
        mma_bf16_ss(tmem + kTmS, smem_desc_sw128(X + off, 16, 1024),
                    smem_desc_sw128(Y + off, 16, 1024), id_qk, kk > 0);
      }
      mma_commit(s_full);
    }
    // every thread waits (bounded); the CTA then agrees on the outcome, so
    // that all threads take the same path through the barriers below
    if (!__syncthreads_and(mbar_wait(s_full, phase, abort))) {
      ok = false;
      break;
    }
    // 2. the value rows into the buffers S no longer reads (they land while
    // the probabilities are computed)
    const __nv_bfloat16* vn = apos >= 0 ? v_new + (((int64_t)b * M_max + a0 + t) * H + h) * kTuD
                                        : nullptr;
    load_row(X, t, vn);
    load_row(Y, t, apos >= 0 ? v + aoff : nullptr);
    // 3. P = 2^(s scale log2 e - lse log2 e) of the row over the pass's columns
    tc_fence_after();
    uint32_t raw[kTuCols];
#pragma unroll
    for (int c = 0; c < kTuCols / 32; ++c)
      tmem_ld_32x32b_x32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&raw[c * 32]));
    tmem_ld_wait();
    const int nvalid = na - a0;  // columns of this pass (> 0); beyond: P = 0
    const float2 sc = make_float2(scale_log2e, scale_log2e), n2 = make_float2(nl, nl);
#pragma unroll
    for (int c = 0; c < kTuCols / 32; ++c) {
      uint32_t pk[16], nk[16];
#pragma unroll
      for (int cc = 0; cc < 16; ++cc) {
        const int j = c * 32 + cc * 2;
        const float2 a = __ffma2_rn(make_float2(__uint_as_float(raw[j]), __uint_as_float(raw[j + 1])),
                                    sc, n2);
        const float e0 = j < nvalid ? ex2_approx(a.x) : 0.f;
        const float e1 = j + 1 < nvalid ? ex2_approx(a.y) : 0.f;
        pk[cc] = pack_bf16x2(e0, e1);
        nk[cc] = pk[cc] ^ 0x80008000u;  // -P: both signs flipped
      }
      tmem_st_32x32b_x16(tS + c * 16, pk);
      tmem_st_32x32b_x16(tS + 64 + c * 16, nk);
    }
    tmem_st_wait();
    cp_async_wait_all();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // 4. O (+)= P V'_A, O += (-P) V_A
    if (t == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTuCols / 16; ++kk)
        mma_bf16_ts(tmem + kTmO, tmem + kTmS + kk * 8,
                    smem_desc_sw128(X + kk * 16 * 128, kTuBox, 1024), id_pv,
                    (a0 > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < kTuCols / 16; ++kk)
        mma_bf16_ts(tmem + kTmO, tmem + kTmS + 64 + kk * 8,
                    smem_desc_sw128(Y + kk * 16 * 128, kTuBox, 1024), id_pv, 1u);
      mma_commit(o_done);
    }
    // the next pass reloads the buffers and overwrites S: wait for these products
    if (!__syncthreads_and(mbar_wait(o_done, phase, abort))) {
      ok = false;
      break;
    }
  }

  // 5. o += the change, on this thread's stable row (float32, rounded once)
  if (ok) {
    tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < kTuD / 32; ++c) {
      uint32_t dv[32];
      tmem_ld_32x32b_x32(tO + c * 32, dv);
      tmem_ld_wait();
      if (pos >= 0) {
        uint4* orow = reinterpret_cast<uint4*>(o + ((int64_t)b * L + pos) * rs +
                                               (int64_t)h * kTuD + c * 32);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 w = orow[u];
          const uint32_t in[4] = {w.x, w.y, w.z, w.w};
          uint32_t out[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            out[e] = pack_bf16x2(bf16_lo(in[e]) + __uint_as_float(dv[u * 8 + 2 * e]),
                                 bf16_hi(in[e]) + __uint_as_float(dv[u * 8 + 2 * e + 1]));
          orow[u] = make_uint4(out[0], out[1], out[2], out[3]);
        }
      }
    }
  } else {
    // a wait ran out: no tensor-core work may still be running when the
    // tensor memory is freed, and no copy may still be landing
    cp_async_wait_all();
    if (t == 0) {
      mma_commit(drained);
      int none = 0;
      mbar_wait(drained, 0, &none);
      report(dev_status, DLLM_ERR_TIMEOUT);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

bool approx_update_tc_supported(int dtype, int d, const void* q, const void* k, const void* v,
                                const void* v_new, const void* o) {
  const auto a16 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  return dtype == DLLM_BF16 && d == kTuD && a16(q) && a16(k) && a16(v) && a16(v_new) && a16(o);
}

cudaError_t launch_approx_update_tc(const void* q, const float* lse, const void* k, const void* v,
                                    const void* v_new, int B, int L, int H, int M_max,
                                    const int32_t* idx, const int32_t* count, int N_max,
                                    const int32_t* stable_idx, const int32_t* stable_count,
                                    float scale, void* o, int32_t* dev_status,
                                    cudaStream_t stream) {
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(approx_update_tc_kernel),
                                    (int)kTuSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((N_max + kTuRows - 1) / kTuRows), (unsigned)H, (unsigned)B);
  launch_pdl(approx_update_tc_kernel, grid, kTuThreads, kTuSmem, stream,
             static_cast<const __nv_bfloat16*>(q), lse, static_cast<const __nv_bfloat16*>(k),
             static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(v_new), idx,
             count, stable_idx, stable_count, static_cast<__nv_bfloat16*>(o), L, H, M_max, N_max,
             scale * kLog2e, dev_status);
  return cudaGetLastError();
}

}  // namespace dllm
