// moe_finalize: top-k weight-and-reduce ("[vLLM] MoE Oracle & Prepare/Finalize"
// blog, "No DP/EP" listing) fused with the single-GPU steps of the flashinfer
// finalize fusion ("[flashinfer] MoE Finalize + AllReduce fusion" page,
// introduction): + shared-expert row, + residual, RMSNorm, optional NVFP4
// packing.  The all-reduce of that fusion has no counterpart on one GPU.
//
// HBM-bound.  One thread-block cluster of kC CTAs owns one token; each CTA
// streams a contiguous 1/kC slice of the row with 16-byte read-only loads.  The
// RMSNorm sum of squares is reduced warp -> CTA -> cluster, the last step over
// distributed shared memory in rank order, so every CTA of the cluster sees the
// same bits.  The shared-expert and residual slices are prefetched into L2 with
// one bulk prefetch each before the expert rows are read, so their latency
// overlaps the k expert-row loads (the shared-row prefetch idea of the
// flashinfer page, "Code analysis", new dispatch tables).
#include <cuda_fp4.h>

#include <algorithm>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
enum OutKind { kOutBF16 = 0, kOutF32 = 1, kOutNVFP4 = 2 };

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Coherent 16-byte load (ld.global.cg): the residual row when the call writes residual_out
// over it (in place), which the read-only path may not be used for.
__device__ __forceinline__ uint4 ldg_cg(const void* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }

__device__ __forceinline__ void add_bf16x8(float (&o)[8], uint4 v, float w) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = fmaf(w, bf16lo(u[i]), o[2 * i]);
    o[2 * i + 1] = fmaf(w, bf16hi(u[i]), o[2 * i + 1]);
  }
}

// 16-byte asynchronous copy global -> shared (L2 only), and the wait for this thread's own
__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_own() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of a cluster barrier phase that orders nothing: arrived at on entry, waited
// on before the first write to another CTA's shared memory (every CTA of the cluster has
// started by then)
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
// Store v at the same shared-memory variable of the cluster's CTA `rank` (distributed shared memory).
__device__ __forceinline__ void st_dsmem_f32(float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Where the expert rows of the slots are: token-major rows y[t * top_k + j] (the standard
// format), or, for the batched format, the row of slot f in an [E, max_tokens, H] output:
// expert e = ids[f], rank inv_slot[f] - offsets[e] among that expert's slots.
struct SlotRows {
  const int32_t* ids;      // NULL: token-major rows
  const int32_t* inv_slot;
  const int32_t* offsets;
  int max_tokens;
  __device__ __forceinline__ size_t row(int t, int top_k, int j) const {
    const int f = t * top_k + j;
    if (!ids) return (size_t)f;
    const int e = __ldg(ids + f);
    return (size_t)e * max_tokens + (__ldg(inv_slot + f) - __ldg(offsets + e));
  }
};

// NV: 16-byte vectors per thread (upper bound); kC: CTAs per token (cluster size).
template <int kC, int NV, int kOut>
__global__ void __launch_bounds__(kThreads)
    finalize_kernel(void* __restrict__ output, const __nv_bfloat16* __restrict__ y, const float* __restrict__ topk_w,
                    const __nv_bfloat16* __restrict__ shared, const __nv_bfloat16* residual,
                    const __nv_bfloat16* __restrict__ gamma, float eps, int H, int top_k, int weights_on_input,
                    uint8_t* __restrict__ out_scale, float gscale, __nv_bfloat16* residual_out,
                    const SlotRows rows) {
  // residual_out may be residual itself (the in-place add + RMSNorm): each element is read
  // by the thread that later writes it, through coherent loads in that case
  const bool res_in_place = residual_out != nullptr && residual_out == residual;
  __shared__ float red[kThreads / 32];
  __shared__ float cta_ss[kC];  // the sum of squares of each CTA of the cluster, by rank
  // the slice of the RMSNorm weight, copied in at the start (no registers held while
  // the rows stream in); each thread reads back only the vectors it copied
  __shared__ __align__(16) uint4 gamma_s[NV * kThreads];
  const int t = blockIdx.x / kC;
  const uint32_t rank = kC > 1 ? cluster_rank() : 0;
  if (kC > 1 && gamma) cluster_arrive_relaxed();
  const int vslice = H / 8 / kC;                // vectors of this CTA's slice
  const int v0 = (int)rank * vslice;            // first vector of the slice within the row
  const size_t row = (size_t)t * H;

  float o[NV][8];
#pragma unroll
  for (int u = 0; u < NV; ++u)
#pragma unroll
    for (int i = 0; i < 8; ++i) o[u][i] = 0.f;

  if (threadIdx.x == 0) {
    // one CTA per token: its expert rows 1..k-1 (row 0 is loaded at once; measured: with
    // clusters, whose slices are short, the extra requests cost more than they save)
    if (kC == 1)
      for (int j = 1; j < top_k; ++j)
        prefetch_l2(y + rows.row(t, top_k, j) * H, (uint32_t)H * 2);
    // then the shared and residual slices
    if (shared) prefetch_l2(shared + row + (size_t)v0 * 8, (uint32_t)vslice * 16);
    if (residual) prefetch_l2(residual + row + (size_t)v0 * 8, (uint32_t)vslice * 16);
  }
  if (gamma) {
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      const int vi = threadIdx.x + u * kThreads;
      if (vi < vslice) cp_async_16(&gamma_s[vi], gamma + (size_t)(v0 + vi) * 8);
    }
  }

  // Short slices (a few vectors per thread, the cluster launches of small T): every row's
  // loads are issued before the first add, so the k + 2 rows cost one memory round trip
  // instead of one each.  The adds keep the row order of the general path (same bits).
  constexpr int kMaxBatchK = 8;
  if (NV <= 2 && top_k <= kMaxBatchK) {
    uint4 yv[kMaxBatchK][NV], sv[NV], rv[NV];
    float wj[kMaxBatchK];
#pragma unroll
    for (int j = 0; j < kMaxBatchK; ++j) {
      if (j < top_k) {
        wj[j] = weights_on_input ? 1.0f : __ldg(topk_w + (size_t)t * top_k + j);
        const __nv_bfloat16* yr = y + rows.row(t, top_k, j) * H + (size_t)v0 * 8;
#pragma unroll
        for (int u = 0; u < NV; ++u) {
          const int vi = threadIdx.x + u * kThreads;
          if (vi < vslice) yv[j][u] = ldg_nc(yr + (size_t)vi * 8);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      const int vi = threadIdx.x + u * kThreads;
      if (shared && vi < vslice) sv[u] = ldg_nc(shared + row + (size_t)(v0 + vi) * 8);
      if (residual && vi < vslice)
        rv[u] = res_in_place ? ldg_cg(residual + row + (size_t)(v0 + vi) * 8)
                             : ldg_nc(residual + row + (size_t)(v0 + vi) * 8);
    }
#pragma unroll
    for (int j = 0; j < kMaxBatchK; ++j)
      if (j < top_k)
#pragma unroll
        for (int u = 0; u < NV; ++u)
          if (threadIdx.x + u * kThreads < vslice) add_bf16x8(o[u], yv[j][u], wj[j]);
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      if (threadIdx.x + u * kThreads >= vslice) continue;
      if (shared) add_bf16x8(o[u], sv[u], 1.0f);
      if (residual) add_bf16x8(o[u], rv[u], 1.0f);
    }
  } else {
    for (int j = 0; j < top_k; ++j) {
      const float w = weights_on_input ? 1.0f : __ldg(topk_w + (size_t)t * top_k + j);
      const __nv_bfloat16* yr = y + rows.row(t, top_k, j) * H + (size_t)v0 * 8;
      uint4 v[NV];
#pragma unroll
      for (int u = 0; u < NV; ++u) {
        const int vi = threadIdx.x + u * kThreads;
        if (vi < vslice) v[u] = ldg_nc(yr + (size_t)vi * 8);
      }
#pragma unroll
      for (int u = 0; u < NV; ++u)
        if (threadIdx.x + u * kThreads < vslice) add_bf16x8(o[u], v[u], w);
    }
    if (shared) {
#pragma unroll
      for (int u = 0; u < NV; ++u) {
        const int vi = threadIdx.x + u * kThreads;
        if (vi < vslice) add_bf16x8(o[u], ldg_nc(shared + row + (size_t)(v0 + vi) * 8), 1.0f);
      }
    }
    if (residual) {
#pragma unroll
      for (int u = 0; u < NV; ++u) {
        const int vi = threadIdx.x + u * kThreads;
        if (vi < vslice)
          add_bf16x8(o[u], res_in_place ? ldg_cg(residual + row + (size_t)(v0 + vi) * 8)
                                        : ldg_nc(residual + row + (size_t)(v0 + vi) * 8), 1.0f);
      }
    }
  }
  if (residual_out) {
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      const int vi = threadIdx.x + u * kThreads;
      if (vi < vslice) {
        uint4 p;
        p.x = pack_bf16x2(o[u][0], o[u][1]);
        p.y = pack_bf16x2(o[u][2], o[u][3]);
        p.z = pack_bf16x2(o[u][4], o[u][5]);
        p.w = pack_bf16x2(o[u][6], o[u][7]);
        *reinterpret_cast<uint4*>(residual_out + row + (size_t)(v0 + vi) * 8) = p;
      }
    }
  }

  if (gamma) {
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u)
      if (threadIdx.x + u * kThreads < vslice)
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(o[u][i], o[u][i], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    if (kC > 1) cluster_wait();  // (the phase arrived at on entry: every peer has started)
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) s += red[w];
      // this CTA's sum goes to slot `rank` of every CTA of the cluster (its own included)
      if (kC > 1) {
#pragma unroll
        for (int r = 0; r < kC; ++r) st_dsmem_f32(&cta_ss[rank], (uint32_t)r, s);
      } else {
        cta_ss[0] = s;
      }
    }
    // one cluster barrier: every slot of every CTA is written (the stores precede the
    // release), and no CTA is read from after it, so each may leave as soon as it is done
    if (kC > 1)
      cluster_sync();
    else
      __syncthreads();
    float total = 0.f;
#pragma unroll
    for (int r = 0; r < kC; ++r) total += cta_ss[r];  // rank order: the same bits in every CTA
    const float inv = rsqrtf(total / (float)H + eps);
    cp_async_wait_own();
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      const int vi = threadIdx.x + u * kThreads;
      if (vi < vslice) {
        const uint4 g = gamma_s[vi];
        const uint32_t gu[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[u][2 * i] = o[u][2 * i] * inv * bf16lo(gu[i]);
          o[u][2 * i + 1] = o[u][2 * i + 1] * inv * bf16hi(gu[i]);
        }
      }
    }
  }

#pragma unroll
  for (int u = 0; u < NV; ++u) {
    const int vi = threadIdx.x + u * kThreads;
    const bool ok = vi < vslice;
    const size_t e0 = row + (size_t)(v0 + vi) * 8;  // first element of this vector
    if (kOut == kOutBF16) {
      if (ok) {
        uint4 p;
        p.x = pack_bf16x2(o[u][0], o[u][1]);
        p.y = pack_bf16x2(o[u][2], o[u][3]);
        p.z = pack_bf16x2(o[u][4], o[u][5]);
        p.w = pack_bf16x2(o[u][6], o[u][7]);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(output) + e0) = p;
      }
    } else if (kOut == kOutF32) {
      if (ok) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(output) + e0);
        dst[0] = make_float4(o[u][0], o[u][1], o[u][2], o[u][3]);
        dst[1] = make_float4(o[u][4], o[u][5], o[u][6], o[u][7]);
      }
    } else {
      // 16-element group = vectors (2m, 2m+1) = this thread and its neighbour
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(o[u][i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      const __nv_fp8_storage_t sf8 = __nv_cvt_float_to_fp8(__fdiv_rn(amax, 6.0f * gscale), __NV_SATFINITE, __NV_E4M3);
      const float sf = __half2float(__half(__nv_cvt_fp8_to_halfraw(sf8, __NV_E4M3)));
      const float denom = sf * gscale;
      uint32_t q = 0;
      if (denom > 0.f) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 r = make_float2(__fdiv_rn(o[u][2 * i], denom), __fdiv_rn(o[u][2 * i + 1], denom));
          q |= (uint32_t)__nv_cvt_float2_to_fp4x2(r, __NV_E2M1, cudaRoundNearest) << (8 * i);
        }
      }
      if (ok) {
        reinterpret_cast<uint32_t*>(output)[e0 / 8] = q;  // 8 codes = 4 bytes
        if ((threadIdx.x & 1) == 0) out_scale[e0 / 16] = (uint8_t)sf8;
      }
    }
  }
}

template <int kC, int NV, int kOut>
cudaError_t launch_finalize(cudaStream_t s, int T, void* output, const void* y, const float* w, const void* shared,
                            const void* residual, const void* gamma, float eps, int H, int top_k, int won,
                            uint8_t* out_scale, float gscale, void* residual_out, const SlotRows& rows) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)T * kC);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, finalize_kernel<kC, NV, kOut>, output,
                            static_cast<const __nv_bfloat16*>(y), w, static_cast<const __nv_bfloat16*>(shared),
                            static_cast<const __nv_bfloat16*>(residual), static_cast<const __nv_bfloat16*>(gamma),
                            eps, H, top_k, won, out_scale, gscale, static_cast<__nv_bfloat16*>(residual_out), rows);
}

template <int kOut>
cudaError_t dispatch_finalize(int C, int nv, cudaStream_t s, int T, void* output, const void* y, const float* w,
                              const void* shared, const void* residual, const void* gamma, float eps, int H,
                              int top_k, int won, uint8_t* out_scale, float gscale, void* residual_out,
                              const SlotRows& rows) {
#define MOE_FIN(CC, NVV)                                                                                       \
  if (C == CC && nv <= NVV)                                                                                    \
    return launch_finalize<CC, NVV, kOut>(s, T, output, y, w, shared, residual, gamma, eps, H, top_k, won, \
                                          out_scale, gscale, residual_out, rows);
  MOE_FIN(1, 2) MOE_FIN(1, 4) MOE_FIN(1, 8)
  MOE_FIN(2, 2) MOE_FIN(2, 4) MOE_FIN(2, 8)
  MOE_FIN(4, 2) MOE_FIN(4, 4) MOE_FIN(4, 8)
#undef MOE_FIN
  return cudaErrorInvalidValue;
}

}  // namespace

MOE_DEFINE_STATUS_READER(finalize_status)

}  // namespace moe

using namespace moe;

namespace {
moe_status_t finalize_run(void* output, const void* fused_expert_output, const float* topk_weights, const void* shared,
                          const void* residual, const void* rms_weight, float eps, int T, int H, int top_k,
                          int apply_router_weight_on_input, moe_dtype_t out_dtype, uint8_t* out_scale,
                          float out_global_scale, void* residual_out, const SlotRows& rows, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && H > 0 && H % 8 == 0 && top_k >= 1 && top_k <= 32);
  MOE_CHECK_ARG(out_dtype == MOE_DT_BF16 || out_dtype == MOE_DT_FP32 || out_dtype == MOE_DT_NVFP4);
  MOE_CHECK_ARG(out_dtype != MOE_DT_NVFP4 || (H % 16 == 0 && out_global_scale > 0.f));
  MOE_CHECK_ARG(fits_int32((long long)T * top_k * (long long)H / 8) && fits_int32((long long)T * 4));
  MOE_CHECK_ARG(eps >= 0.f);
  if (T == 0) return MOE_OK;
  MOE_CHECK_ARG(output && fused_expert_output && aligned16(output) && aligned16(fused_expert_output));
  MOE_CHECK_ARG(apply_router_weight_on_input || topk_weights);
  MOE_CHECK_ARG(out_dtype != MOE_DT_NVFP4 || out_scale);
  MOE_CHECK_ARG(aligned16(shared) && aligned16(residual) && aligned16(rms_weight) && aligned16(residual_out));
  // Cluster size: the smallest of 1, 2, 4 whose row slices fit one CTA's
  // registers (8 vectors per thread), grown while the grid has fewer than 4
  // CTAs per SM (measured: T=512 at H=7168 is 3% faster with 2-CTA clusters
  // than with one CTA per token).  With NVFP4 output the slices are whole
  // 16-element groups.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int won = apply_router_weight_on_input ? 1 : 0;
  cudaError_t err;
  const int nsm = num_sms();
  const int grp = out_dtype == MOE_DT_NVFP4 ? 16 : 8;
  auto slice_ok = [&](int c) { return H % (grp * c) == 0 && (H / 8) / c <= 8 * kThreads; };
  int C = 1;
  while (C < 4 && !slice_ok(C)) C *= 2;
  if (!slice_ok(C)) return MOE_ERR_UNSUPPORTED;
  while (C < 4 && (long long)T * C < 4LL * nsm && slice_ok(2 * C) && (H / 8) / (2 * C) >= kThreads) C *= 2;
  const int per_cta = (H / 8) / C;
  const int nv = (per_cta + kThreads - 1) / kThreads;
  if (out_dtype == MOE_DT_BF16)
    err = dispatch_finalize<kOutBF16>(C, nv, s, T, output, fused_expert_output, topk_weights, shared, residual,
                                      rms_weight, eps, H, top_k, won, out_scale, out_global_scale, residual_out, rows);
  else if (out_dtype == MOE_DT_FP32)
    err = dispatch_finalize<kOutF32>(C, nv, s, T, output, fused_expert_output, topk_weights, shared, residual,
                                     rms_weight, eps, H, top_k, won, out_scale, out_global_scale, residual_out, rows);
  else
    err = dispatch_finalize<kOutNVFP4>(C, nv, s, T, output, fused_expert_output, topk_weights, shared, residual,
                                       rms_weight, eps, H, top_k, won, out_scale, out_global_scale, residual_out, rows);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  return launch_status();
}
}  // namespace

extern "C" moe_status_t moe_finalize(void* output, const void* fused_expert_output, const float* topk_weights,
                                     const int32_t* topk_ids, const void* shared, const void* residual,
                                     const void* rms_weight, float eps, int T, int H, int top_k,
                                     int apply_router_weight_on_input, moe_dtype_t out_dtype, uint8_t* out_scale,
                                     float out_global_scale, void* residual_out, moe_stream_t stream) {
  (void)topk_ids;
  const SlotRows rows{nullptr, nullptr, nullptr, 0};
  return finalize_run(output, fused_expert_output, topk_weights, shared, residual, rms_weight, eps, T, H, top_k,
                      apply_router_weight_on_input, out_dtype, out_scale, out_global_scale, residual_out, rows, stream);
}

extern "C" moe_status_t moe_finalize_batched(void* output, const void* expert_output_b, int max_tokens,
                                             const float* topk_weights, const int32_t* topk_ids,
                                             const int32_t* inv_slot, const int32_t* expert_offsets, const void* shared,
                                             const void* residual, const void* rms_weight, float eps, int T, int H,
                                             int top_k, int apply_router_weight_on_input, moe_dtype_t out_dtype,
                                             uint8_t* out_scale, float out_global_scale, void* residual_out,
                                             moe_stream_t stream) {
  MOE_CHECK_ARG(max_tokens >= 1);
  if (T > 0) MOE_CHECK_ARG(topk_ids && inv_slot && expert_offsets);
  const SlotRows rows{topk_ids, inv_slot, expert_offsets, max_tokens};
  return finalize_run(output, expert_output_b, topk_weights, shared, residual, rms_weight, eps, T, H, top_k,
                      apply_router_weight_on_input, out_dtype, out_scale, out_global_scale, residual_out, rows, stream);
}
