// moe_route: top-k router, one warp per token.
//
// The pages pass topk_ids / topk_weights into prepare and finalize ("[vLLM] MoE
// Oracle & Prepare/Finalize" blog, "No DP/EP" listing) without defining the
// router; this kernel computes the plain reading: the top_k largest logits
// (ties to the lower expert index) with softmax weights renormalised over the
// chosen experts, or top-1 with a sigmoid weight for the Llama-type router that
// applies its weight on the input ("Fused MoE Kernel Features", All2All
// section).
//
// Each lane holds E/32 logits in registers; every round is a lane-local argmax
// followed by a 5-step butterfly argmax across the warp, so the selected order
// and ids are exact and independent of scheduling.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

template <int NV>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_kernel(const float* __restrict__ logits, int T, int E, int top_k, int scoring,
                 int32_t* __restrict__ topk_ids, float* __restrict__ topk_weights) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
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
      if (!((taken >> i) & 1u) && better(v[i], idx, bv, bi)) {
        bv = v[i];
        bi = idx;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (better(ov, oi, bv, bi)) {
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

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_route(const float* logits, int T, int E, int top_k, int scoring,
                                  int32_t* topk_ids, float* topk_weights, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && E >= 1 && E <= 1024 && top_k >= 1 && top_k <= E && top_k <= 32);
  MOE_CHECK_ARG(scoring == MOE_SCORING_SOFTMAX_RENORM || scoring == MOE_SCORING_SIGMOID);
  MOE_CHECK_ARG(scoring != MOE_SCORING_SIGMOID || top_k == 1);
  MOE_CHECK_ARG(fits_int32((long long)T * E) && fits_int32((long long)T * top_k));
  if (T == 0) return MOE_OK;
  MOE_CHECK_ARG(logits && topk_ids && topk_weights);
  const dim3 grid((T + kWarpsPerBlock - 1) / kWarpsPerBlock), block(kWarpsPerBlock * 32);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int nv = (E + 31) / 32;
  if (nv <= 1)
    route_kernel<1><<<grid, block, 0, s>>>(logits, T, E, top_k, scoring, topk_ids, topk_weights);
  else if (nv <= 2)
    route_kernel<2><<<grid, block, 0, s>>>(logits, T, E, top_k, scoring, topk_ids, topk_weights);
  else if (nv <= 4)
    route_kernel<4><<<grid, block, 0, s>>>(logits, T, E, top_k, scoring, topk_ids, topk_weights);
  else if (nv <= 8)
    route_kernel<8><<<grid, block, 0, s>>>(logits, T, E, top_k, scoring, topk_ids, topk_weights);
  else if (nv <= 16)
    route_kernel<16><<<grid, block, 0, s>>>(logits, T, E, top_k, scoring, topk_ids, topk_weights);
  else
    route_kernel<32><<<grid, block, 0, s>>>(logits, T, E, top_k, scoring, topk_ids, topk_weights);
  return launch_status();
}
