// refine_common.cuh -- the per-token part of HubKV's refinement (HubKV
// walkthrough, Method: 最终算法, steps 1, 2 and 4), shared by the refinement's
// apply kernel and the fused refine + Top-K kernel so that both produce the
// same z bit for bit.
#pragma once

#include <cmath>

namespace kvc {

// z_i from the window of scores around token i.  `win` points at s_i inside a
// buffer that holds s_{i-half} .. s_{i+half}, with -inf where the window passes
// an end of the prompt [0, T).
//   local hubs (default): q_i = s_i if s_i is the window maximum, gamma s_i otherwise;
//   AVG (KV_HUB_AVGPOOL): q_i = the mean of the window cut at the ends, summed in
//   window order;
// then the ratio gate z_i = s_i + r^2 (beta q_i - s_i).
template <bool AVG>
__device__ __forceinline__ float hub_gate(const float *win, int half, int i, int T, float gamma, float r2,
                                          float beta) {
  const float si = win[0];
  float qi;
  if constexpr (AVG) {
    float sum = 0.f;
    int cnt = 0;
    for (int o = -half; o <= half; ++o)
      if (i + o >= 0 && i + o < T) {
        sum += win[o];
        ++cnt;
      }
    qi = sum / (float)cnt;
  } else {
    float M = si;
    for (int o = -half; o <= half; ++o) M = fmaxf(M, win[o]);
    qi = (si == M) ? si : gamma * si;
  }
  return fmaf(r2, fmaf(beta, qi, -si), si);  // s + r^2 (beta q - s)
}

}  // namespace kvc
