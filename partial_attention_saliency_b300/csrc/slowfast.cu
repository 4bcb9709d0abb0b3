// SlowFast phase control: host-side state of the sampler's slow/fast cycle.
//
// SlowFast ("Accelerating Diffusion Large Language Models with SlowFast
// Sampling: The Three Golden Principles"), section 2 (pipeline): the slow
// phase watches the prediction of the convergence point e_cand over a sliding
// window of steps; once the variance of the prediction falls below
// sigma^2_stable the region [s_cycle, e_cycle] is stable and the fast phase
// decodes it; then a new cycle begins.
//
// Per batch row the controller keeps the predictions of the current cycle
// (at most `window` of them).  A step is fast iff the window is full, its
// latest prediction lies beyond the start, and the population variance is
// below sigma^2, evaluated exactly on the integers as
// W sum x^2 - (sum x)^2 < sigma^2 W^2 (the right side in double).  A fast step
// returns the region end (the latest prediction) and empties the window.
// Everything here runs on the host; the predictions themselves come from the
// device (the stable-prefix length of the confidence scores from the start).
#include <cstdint>
#include <deque>
#include <new>
#include <vector>

#include "dllm.h"
#include "internal.h"

struct dllm_slowfast {
  int B = 0;
  int window = 0;
  double sigma2 = 0.0;
  std::vector<std::deque<int64_t>> hist;
};

extern "C" dllm_status dllm_slowfast_create(int B, int window, double sigma2_stable,
                                            dllm_slowfast** out) {
  if (out == nullptr)
    return (dllm_status)dllm::set_last_error(DLLM_ERR_INVALID_ARG,
                                             "dllm_slowfast_create: NULL output pointer");
  *out = nullptr;
  if (B < 1 || window < 1 || !(sigma2_stable >= 0.0))
    return (dllm_status)dllm::set_last_error(
        DLLM_ERR_INVALID_ARG, "dllm_slowfast_create: B, window must be >= 1, sigma2 >= 0");
  dllm_slowfast* sf = new (std::nothrow) dllm_slowfast;
  if (sf == nullptr)
    return (dllm_status)dllm::set_last_error(DLLM_ERR_INVALID_ARG,
                                             "dllm_slowfast_create: out of host memory");
  sf->B = B;
  sf->window = window;
  sf->sigma2 = sigma2_stable;
  sf->hist.assign((size_t)B, std::deque<int64_t>());
  *out = sf;
  return DLLM_OK;
}

extern "C" dllm_status dllm_slowfast_observe(dllm_slowfast* sf, const int32_t* start,
                                             const int32_t* e_cand, int32_t* phase_out,
                                             int32_t* region_end_out) {
  if (sf == nullptr || start == nullptr || e_cand == nullptr || phase_out == nullptr ||
      region_end_out == nullptr)
    return (dllm_status)dllm::set_last_error(DLLM_ERR_INVALID_ARG,
                                             "dllm_slowfast_observe: NULL pointer argument");
  const int64_t W = sf->window;
  for (int b = 0; b < sf->B; ++b) {
    std::deque<int64_t>& h = sf->hist[(size_t)b];
    h.push_back(e_cand[b]);
    if ((int64_t)h.size() > W) h.pop_front();
    phase_out[b] = 0;
    region_end_out[b] = -1;
    if ((int64_t)h.size() == W && h.back() > start[b]) {
      int64_t s1 = 0, s2 = 0;
      for (int64_t x : h) {
        s1 += x;
        s2 += x * x;
      }
      const int64_t num = W * s2 - s1 * s1;  // W^2 times the population variance
      if ((double)num < sf->sigma2 * (double)(W * W)) {
        phase_out[b] = 1;
        region_end_out[b] = (int32_t)h.back();
        h.clear();
      }
    }
  }
  return DLLM_OK;
}

extern "C" void dllm_slowfast_destroy(dllm_slowfast* sf) { delete sf; }
