// Router arithmetic shared by the route kernel and the single-launch layer: one
// warp per token.  Each lane holds E/32 logits in registers; every round is a
// lane-local argmax followed by a 5-step butterfly argmax across the warp, so the
// selected order and ids are exact and independent of scheduling.
#pragma once
#include "moe_common.cuh"

namespace moe {

__device__ __forceinline__ bool route_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Token t's top_k experts and weights, computed by one whole warp.
template <int NV>
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int t, int E, int top_k, int scoring,
                                            int32_t* __restrict__ topk_ids, float* __restrict__ topk_weights) {
  const int lane = threadIdx.x & 31;
  const float* row = logits + (size_t)t * E;

  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = lane + 32 * i;
    float x = idx < E ? __ldg(row + idx) : -INFINITY;
    v[i] = (x != x) ? -INFINITY : x;  // NaN ranks below every number
  }
  uint32_t taken = 0;  // bit i: expert lane + 32 i already chosen (or absent)
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (lane + 32 * i >= E) taken |= 1u << i;

  float my_v = 0.f;  // lane j < top_k keeps the j-th choice
  int my_i = 0;
  for (int r = 0; r < top_k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = lane + 32 * i;
      if (!((taken >> i) & 1u) && route_better(v[i], idx, bv, bi)) {
        bv = v[i];
        bi = idx;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (route_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == r) {
      my_v = bv;
      my_i = bi;
    }
  }

  float w;
  if (scoring == MOE_SCORING_SIGMOID) {
    w = __fdiv_rn(1.0f, 1.0f + expf(-my_v));
  } else {
    const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
    const float e = lane < top_k ? expf(my_v - vmax) : 0.f;
    float s = e;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    w = __fdiv_rn(e, s);
  }
  if (lane < top_k) {
    topk_ids[(size_t)t * top_k + lane] = my_i;
    topk_weights[(size_t)t * top_k + lane] = w;
  }
}


}  // namespace moe
