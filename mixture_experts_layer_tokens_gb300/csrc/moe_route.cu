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
// The per-token arithmetic (one warp per token) is in moe_route.cuh.
#include "moe_route.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

template <int NV>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_kernel(const float* __restrict__ logits, int T, int E, int top_k, int scoring,
                 int32_t* __restrict__ topk_ids, float* __restrict__ topk_weights) {
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  route_token<NV>(logits, t, E, top_k, scoring, topk_ids, topk_weights);
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
