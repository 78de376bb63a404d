// moe_prepare: the prepare step of the no-DP/EP pipeline ("[vLLM] MoE Oracle &
// Prepare/Finalize" blog, "No DP/EP" listing): optional top-k weight on the
// input (top_k == 1), then input quantisation -- bf16 passthrough, or fp8 E4M3
// with one fp32 scale per token per 128 channels (the "G(128)" format of the
// "Fused MoE Kernel Features" tables).
//
// HBM-bound: each thread moves one 16-byte vector of 8 bf16 values; the 16
// threads of a 128-channel group reduce their amax with shuffles.  The scale
// and the codes use IEEE division (never a reciprocal multiply) so the codes
// are exactly those of the definition.
//
// The "A" (per token) and "T" (per tensor) formats of the same tables use the
// same rule over a whole row or the whole tensor: a block per token reduces the
// row's amax and then quantises the row (read twice, the second time from L2);
// the tensor format reduces block amaxes with one atomicMax on the scale word
// (non-negative floats order like their bit patterns), quantises, and a last
// one-thread launch turns that amax into the scale.
#include <algorithm>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;


__device__ __forceinline__ void apply_weight(float (&x)[8], const float* topk_weights, int t) {
  // a1 * topk_weights.to(a1.dtype): the weight is rounded to bf16 first; the
  // product of two bf16 numbers is exact in fp32 and is rounded once to bf16.
  const float wb = __bfloat162float(__float2bfloat16_rn(__ldg(topk_weights + t)));
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = __bfloat162float(__float2bfloat16_rn(x[i] * wb));
}

template <bool kWeight>
__global__ void __launch_bounds__(kThreads)
    prepare_bf16_kernel(const __nv_bfloat16* __restrict__ a1, const float* __restrict__ topk_weights, int H,
                        long long nvec, __nv_bfloat16* __restrict__ a1q) {
  const long long v = (long long)blockIdx.x * kThreads + threadIdx.x;
  if (v >= nvec) return;
  const int vec_per_row = H / 8;
  const int t = (int)(v / vec_per_row);
  float x[8];
  load_bf16x8(a1 + v * 8, x);
  if (kWeight) apply_weight(x, topk_weights, t);
  uint4 o;
  o.x = pack_bf16x2(x[0], x[1]);
  o.y = pack_bf16x2(x[2], x[3]);
  o.z = pack_bf16x2(x[4], x[5]);
  o.w = pack_bf16x2(x[6], x[7]);
  reinterpret_cast<uint4*>(a1q)[v] = o;
}

// One 128-channel group = 16 consecutive threads (half a warp).
template <bool kWeight>
__global__ void __launch_bounds__(kThreads)
    prepare_fp8_kernel(const __nv_bfloat16* __restrict__ a1, const float* __restrict__ topk_weights, int H,
                       long long nvec, uint8_t* __restrict__ a1q, float* __restrict__ a1q_scale) {
  const long long v = (long long)blockIdx.x * kThreads + threadIdx.x;
  // nvec is a multiple of 16, so a half warp is either fully in range or fully out
  if (v >= nvec) return;
  const int vec_per_row = H / 8;
  const int t = (int)(v / vec_per_row);
  float x[8];
  load_bf16x8(a1 + v * 8, x);
  if (kWeight) apply_weight(x, topk_weights, t);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const unsigned half_mask = (threadIdx.x & 16) ? 0xffff0000u : 0x0000ffffu;
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(half_mask, amax, off));
  const float s = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
  const float rs = __frcp_rn(s);
  uint32_t packed[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 r = make_float2(div_rn_by(x[2 * i], s, rs), div_rn_by(x[2 * i + 1], s, rs));
    const uint32_t two = (uint32_t)__nv_cvt_float2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3);
    if (i & 1)
      packed[i >> 1] |= two << 16;
    else
      packed[i >> 1] = two;
  }
  reinterpret_cast<uint2*>(a1q)[v] = make_uint2(packed[0], packed[1]);
  if ((threadIdx.x & 15) == 0) a1q_scale[v / 16] = s;  // [T, H/128] row-major == group index
}




// "A": block t quantises token t with one scale over its H channels.
template <bool kWeight>
__global__ void __launch_bounds__(kThreads)
    prepare_fp8_token_kernel(const __nv_bfloat16* __restrict__ a1, const float* __restrict__ topk_weights, int H,
                             uint8_t* __restrict__ a1q, float* __restrict__ a1q_scale) {
  const int t = blockIdx.x;
  const int nv = H / 8;
  const __nv_bfloat16* row = a1 + (size_t)t * H;
  float a = 0.f;
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    float x[8];
    load_bf16x8(row + (size_t)v * 8, x);
    if (kWeight) apply_weight(x, topk_weights, t);
    a = fmaxf(a, amax8(x));
  }
  const float s = __fdiv_rn(fmaxf(block_amax<kThreads>(a), 1e-10f), 448.0f);
  uint2* out = reinterpret_cast<uint2*>(a1q + (size_t)t * H);
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    float x[8];
    load_bf16x8(row + (size_t)v * 8, x);
    if (kWeight) apply_weight(x, topk_weights, t);
    out[v] = e4m3x8(x, s);
  }
  if (threadIdx.x == 0) a1q_scale[t] = s;
}

// "T", step 1: amax of the tensor into *amax_bits (zeroed before the launch).
template <bool kWeight>
__global__ void __launch_bounds__(kThreads)
    prepare_fp8_tensor_amax_kernel(const __nv_bfloat16* __restrict__ a1, const float* __restrict__ topk_weights,
                                   int H, long long nvec, unsigned* __restrict__ amax_bits) {
  const int vpr = H / 8;
  float a = 0.f;
  for (long long v = (long long)blockIdx.x * kThreads + threadIdx.x; v < nvec; v += (long long)gridDim.x * kThreads) {
    float x[8];
    load_bf16x8(a1 + v * 8, x);
    if (kWeight) apply_weight(x, topk_weights, (int)(v / vpr));
    a = fmaxf(a, amax8(x));
  }
  a = block_amax<kThreads>(a);
  if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(a));
}

// "T", step 2: codes with s = fp32(max(amax, 1e-10) / 448).
template <bool kWeight>
__global__ void __launch_bounds__(kThreads)
    prepare_fp8_tensor_kernel(const __nv_bfloat16* __restrict__ a1, const float* __restrict__ topk_weights, int H,
                              long long nvec, const unsigned* __restrict__ amax_bits, uint8_t* __restrict__ a1q) {
  const long long v = (long long)blockIdx.x * kThreads + threadIdx.x;
  if (v >= nvec) return;
  const float s = __fdiv_rn(fmaxf(__uint_as_float(*amax_bits), 1e-10f), 448.0f);
  float x[8];
  load_bf16x8(a1 + v * 8, x);
  if (kWeight) apply_weight(x, topk_weights, (int)(v / (H / 8)));
  reinterpret_cast<uint2*>(a1q)[v] = e4m3x8(x, s);
}

// "T", step 3: the amax word becomes the scale.
__global__ void prepare_fp8_tensor_scale_kernel(float* a1q_scale) {
  a1q_scale[0] = __fdiv_rn(fmaxf(a1q_scale[0], 1e-10f), 448.0f);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_prepare(const void* a1, const float* topk_weights, const int32_t* topk_ids, int T, int H,
                                    int top_k, int apply_router_weight_on_input, const moe_quant_config* qc,
                                    void* a1q, float* a1q_scale, moe_stream_t stream) {
  (void)topk_ids;
  MOE_CHECK_ARG(qc && T >= 0 && H > 0 && top_k >= 1);
  MOE_CHECK_ARG(!apply_router_weight_on_input || top_k == 1);  // the pages' `assert topk == 1`
  const bool fp8 = qc->act == MOE_DT_FP8_E4M3;
  if (!fp8 && qc->act != MOE_DT_BF16) return MOE_ERR_UNSUPPORTED;
  if (fp8 && qc->act_group != 128 && qc->act_group != MOE_GROUP_TOKEN && qc->act_group != MOE_GROUP_TENSOR)
    return MOE_ERR_UNSUPPORTED;
  MOE_CHECK_ARG(fp8 ? H % 128 == 0 : H % 8 == 0);
  MOE_CHECK_ARG(fits_int32((long long)T * H / 8 + kThreads));
  if (T == 0) return MOE_OK;
  MOE_CHECK_ARG(a1 && a1q && aligned16(a1) && aligned16(a1q));
  MOE_CHECK_ARG(!apply_router_weight_on_input || topk_weights);
  MOE_CHECK_ARG(!fp8 || a1q_scale);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long nvec = (long long)T * H / 8;
  const unsigned grid = (unsigned)((nvec + kThreads - 1) / kThreads);
  const auto* x = static_cast<const __nv_bfloat16*>(a1);
  if (!fp8) {
    if (!apply_router_weight_on_input) {
      if (a1q == a1) return MOE_OK;  // no quantisation type: the input passes through
      if (cudaMemcpyAsync(a1q, a1, (size_t)T * H * 2, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
      return MOE_OK;
    }
    prepare_bf16_kernel<true><<<grid, kThreads, 0, s>>>(x, topk_weights, H, nvec, static_cast<__nv_bfloat16*>(a1q));
  } else if (qc->act_group == MOE_GROUP_TOKEN) {
    if (apply_router_weight_on_input)
      prepare_fp8_token_kernel<true><<<T, kThreads, 0, s>>>(x, topk_weights, H, static_cast<uint8_t*>(a1q), a1q_scale);
    else
      prepare_fp8_token_kernel<false><<<T, kThreads, 0, s>>>(x, topk_weights, H, static_cast<uint8_t*>(a1q), a1q_scale);
  } else if (qc->act_group == MOE_GROUP_TENSOR) {
    unsigned* amax = reinterpret_cast<unsigned*>(a1q_scale);
    if (cudaMemsetAsync(amax, 0, sizeof(unsigned), s) != cudaSuccess) return MOE_ERR_CUDA;
    const unsigned agrid = (unsigned)std::min<long long>(grid, 4LL * num_sms());
    if (apply_router_weight_on_input) {
      prepare_fp8_tensor_amax_kernel<true><<<agrid, kThreads, 0, s>>>(x, topk_weights, H, nvec, amax);
      prepare_fp8_tensor_kernel<true><<<grid, kThreads, 0, s>>>(x, topk_weights, H, nvec, amax, static_cast<uint8_t*>(a1q));
    } else {
      prepare_fp8_tensor_amax_kernel<false><<<agrid, kThreads, 0, s>>>(x, topk_weights, H, nvec, amax);
      prepare_fp8_tensor_kernel<false><<<grid, kThreads, 0, s>>>(x, topk_weights, H, nvec, amax, static_cast<uint8_t*>(a1q));
    }
    prepare_fp8_tensor_scale_kernel<<<1, 1, 0, s>>>(a1q_scale);
  } else if (apply_router_weight_on_input) {
    prepare_fp8_kernel<true><<<grid, kThreads, 0, s>>>(x, topk_weights, H, nvec, static_cast<uint8_t*>(a1q), a1q_scale);
  } else {
    prepare_fp8_kernel<false><<<grid, kThreads, 0, s>>>(x, topk_weights, H, nvec, static_cast<uint8_t*>(a1q), a1q_scale);
  }
  return launch_status();
}

// ------------------------------------------------------------------ batched activation format
// The batched prepare ("Fused MoE Kernel Features", section "Fused MoE Modular All2All
// backends": the prepare output is "standard" or "batched"): the standard prepare of every
// token into the workspace, then one warp per sorted row p places the prepared row of its
// token in the slab of its expert, at rank p - expert_offsets[e] (the expert's slots in
// ascending order, as moe_align sorts them).  A row whose rank reaches max_tokens is left
// out and MOE_ERR_INVALID_ARG is recorded in the status word.
namespace moe {
namespace {

// Expert of sorted row p: the last e with offsets[e] <= p (offsets ascending, offsets[E] = S).
__device__ __forceinline__ int expert_of_row(const int32_t* __restrict__ offsets, int E, int p) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(offsets + mid) <= p)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// row_bytes: bytes of one prepared row; nscale: fp32 scales per row (G(128): H/128, "A": 1,
// bf16 and "T": 0 -- the tensor scale is copied once).
__global__ void __launch_bounds__(256)
    dispatch_batched_kernel(const uint8_t* __restrict__ a1q, const float* __restrict__ a1q_scale,
                            const int32_t* __restrict__ offsets, const int32_t* __restrict__ sorted_slot, int S,
                            int top_k, int E, int max_tokens, int row_bytes, int nscale, int tensor_scale,
                            uint8_t* __restrict__ a1q_b, float* __restrict__ a1q_b_scale,
                            int32_t* __restrict__ expert_num_tokens) {
  const int gtid = blockIdx.x * 256 + threadIdx.x;
  if (gtid < E) expert_num_tokens[gtid] = min(__ldg(offsets + gtid + 1) - __ldg(offsets + gtid), max_tokens);
  if (gtid == 0 && tensor_scale) a1q_b_scale[0] = __ldg(a1q_scale);
  const int p = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (p >= S) return;
  const int e = expert_of_row(offsets, E, p);
  const int m = p - __ldg(offsets + e);
  if (m >= max_tokens) {
    if (lane == 0) record_status((int)MOE_ERR_INVALID_ARG);
    return;
  }
  const int t = __ldg(sorted_slot + p) / top_k;
  const size_t dst_row = (size_t)e * max_tokens + m;
  const uint4* src = reinterpret_cast<const uint4*>(a1q + (size_t)t * row_bytes);
  uint4* dst = reinterpret_cast<uint4*>(a1q_b + dst_row * row_bytes);
  for (int i = lane; i < row_bytes / 16; i += 32) dst[i] = __ldg(src + i);
  for (int g = lane; g < nscale; g += 32) a1q_b_scale[dst_row * nscale + g] = __ldg(a1q_scale + (size_t)t * nscale + g);
}

size_t batched_prepare_ws(int T, int H, const moe_quant_config* qc, size_t* scale_off) {
  const bool fp8 = qc->act == MOE_DT_FP8_E4M3;
  const size_t codes = (((size_t)T * H * (fp8 ? 1 : 2)) + 255) & ~size_t(255);
  size_t scales = 0;
  if (fp8) scales = qc->act_group == 128 ? (size_t)T * (H / 128) * 4 : (qc->act_group == MOE_GROUP_TOKEN ? (size_t)T * 4 : 16);
  *scale_off = codes;
  return codes + ((scales + 255) & ~size_t(255));
}

}  // namespace

MOE_DEFINE_STATUS_READER(prepare_status)

}  // namespace moe

using namespace moe;

extern "C" size_t moe_prepare_batched_workspace_size(int T, int H, const moe_quant_config* qc) {
  if (!qc || T < 0 || H <= 0) return 0;
  size_t so = 0;
  return std::max<size_t>(batched_prepare_ws(T, H, qc, &so), 256);
}

extern "C" moe_status_t moe_prepare_batched(const void* a1, const float* topk_weights, const int32_t* expert_offsets,
                                            const int32_t* sorted_slot, int T, int H, int top_k, int E,
                                            int max_tokens, int apply_router_weight_on_input,
                                            const moe_quant_config* qc, void* a1q_b, float* a1q_b_scale,
                                            int32_t* expert_num_tokens, void* ws, size_t ws_bytes,
                                            moe_stream_t stream) {
  MOE_CHECK_ARG(qc && T >= 0 && H > 0 && top_k >= 1 && E >= 1 && E <= 1024 && top_k <= E && max_tokens >= 1);
  const bool fp8 = qc->act == MOE_DT_FP8_E4M3;
  MOE_CHECK_ARG(fits_int32((long long)T * top_k) && fits_int32((long long)E * max_tokens) &&
                fits_int32((long long)E * max_tokens * (H / 8)));
  MOE_CHECK_ARG(expert_num_tokens && a1q_b && aligned16(a1q_b) && (!fp8 || a1q_b_scale));
  size_t scale_off = 0;
  size_t need = batched_prepare_ws(T, H, qc, &scale_off);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {  // every expert empty
    return cudaMemsetAsync(expert_num_tokens, 0, (size_t)E * 4, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  MOE_CHECK_ARG(expert_offsets && sorted_slot);
  if (!fp8 && !apply_router_weight_on_input) need = 0;
  if (need && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  MOE_CHECK_ARG(!need || aligned16(ws));
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* sc = fp8 ? reinterpret_cast<float*>(wsb + scale_off) : nullptr;
  // (bf16 without the weight on the input: the rows are a1 itself, placed straight from it)
  const bool direct = !fp8 && !apply_router_weight_on_input;
  MOE_CHECK_ARG(a1 && aligned16(a1));
  if (!direct) {
    const moe_status_t st = moe_prepare(a1, topk_weights, nullptr, T, H, top_k, apply_router_weight_on_input, qc,
                                        wsb, sc, stream);
    if (st != MOE_OK) return st;
  }
  const uint8_t* rows = direct ? static_cast<const uint8_t*>(a1) : wsb;
  const int S = T * top_k;
  const int nscale = !fp8 ? 0 : (qc->act_group == 128 ? H / 128 : (qc->act_group == MOE_GROUP_TOKEN ? 1 : 0));
  const int tensor = fp8 && qc->act_group == MOE_GROUP_TENSOR;
  const unsigned grid = (unsigned)std::max<long long>((S + 7) / 8, (E + 255) / 256);
  dispatch_batched_kernel<<<grid, 256, 0, s>>>(rows, sc, expert_offsets, sorted_slot, S, top_k, E, max_tokens,
                                               H * (fp8 ? 1 : 2), nscale, tensor, static_cast<uint8_t*>(a1q_b),
                                               a1q_b_scale, expert_num_tokens);
  return launch_status();
}
