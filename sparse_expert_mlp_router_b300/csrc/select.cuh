// Warp-level score function + top-k selection for one token.
//
// Scores [shubhamtatvamasi.com/llm-inference/moe "Mixture of Experts", section
// "The router"]: softmax over all E logits (max-subtracted), or the sigmoid
// variant. Selection: the k highest scores in rank order, equal scores to the
// lower expert id; NaN scores rank below every number so a token always gets
// k distinct ids. Gates: the selected scores divided by their sum (or the raw
// scores when renormalisation is off).
#pragma once

#include <cfloat>
#include "internal.cuh"

namespace moe {

__device__ __forceinline__ bool ranks_before(float a, int ea, float b, int eb) {
  return a > b || (a == b && ea < eb);
}

// logits: E values in shared or global memory. Lane l handles experts l, l+32, ...
// Writes idx[0..k), gate[0..k) and, if scores != nullptr, scores[0..E).
__device__ __forceinline__ void select_topk_warp(const float* logits, int E, int k, int score, int renorm,
                                                 int lane, int32_t* idx, float* gate, float* scores) {
  constexpr int kPer = kMaxExperts / 32;
  float s[kPer];
  float mx = -FLT_MAX;
#pragma unroll
  for (int m = 0; m < kPer; ++m) {
    const int e = lane + 32 * m;
    s[m] = (e < E) ? logits[e] : -FLT_MAX;
    if (e < E) mx = fmaxf(mx, s[m]);
  }
  if (score == MOE_SOFTMAX) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int e = lane + 32 * m;
      s[m] = (e < E) ? expf(s[m] - mx) : 0.f;
      sum += s[m];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
#pragma unroll
    for (int m = 0; m < kPer; ++m) s[m] = __fdiv_rn(s[m], sum);
  } else {
#pragma unroll
    for (int m = 0; m < kPer; ++m) s[m] = 1.0f / (1.0f + expf(-s[m]));
  }
  if (scores) {
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int e = lane + 32 * m;
      if (e < E) scores[e] = s[m];
    }
  }
  // selection keys: NaN -> -inf, padding lanes -> -inf with an id past E
  float key[kPer];
#pragma unroll
  for (int m = 0; m < kPer; ++m) {
    const int e = lane + 32 * m;
    key[m] = (e < E && !isnan(s[m])) ? s[m] : -INFINITY;
  }
  unsigned taken = 0;
  float sel[kMaxTopK];
  int sel_e[kMaxTopK];
  float total = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j >= k) break;
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int e = lane + 32 * m;
      if (!(taken >> m & 1u) && e < E && ranks_before(key[m], e, bv, be)) {
        bv = key[m];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ranks_before(ov, oe, bv, be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    // the chosen expert's real score (NaN stays NaN in the gate)
    float sv = 0.f;
#pragma unroll
    for (int m = 0; m < kPer; ++m)
      if (lane + 32 * m == be) sv = s[m];
    sv = __shfl_sync(0xffffffffu, sv, be & 31);
    sel[j] = sv;
    sel_e[j] = be;
    total += sv;
  }
  if (lane == 0) {
    for (int j = 0; j < k; ++j) {
      idx[j] = sel_e[j];
      gate[j] = renorm ? __fdiv_rn(sel[j], total) : sel[j];
    }
  }
}

}  // namespace moe
