// moe_experts: grouped expert MLPs on tcgen05 tensor cores.
//
// "Fused MoE Kernel Features" (vLLM design doc), section "Fused Experts
// Kernels": every expert runs two GEMMs with an activation between them
// (SiLU-and-mul, the SwiGLU default), consumes the prepared (possibly
// quantised) activations and writes its rows in the original activation type.
// For the fp8 G(128) format each token carries one scale per 128 channels and
// each weight one scale per 128x128 block.
//
// Three launches on the caller's stream:
//   gather : a1q rows -> A rows in expert order (sorted_slot), fp8 scales
//            transposed to [K/128][rows]; skipped for the bf16 identity case
//   gemm1  : h = silu(A w13_g^T) * (A w13_u^T), bf16 or fp8 G(128) requantised
//   gemm2  : y[sorted_slot[p]] = h_p w2^T, bf16 rows scattered token-major
//
// GEMM design (one persistent CTA per SM, 128 x 256 output tile per work item):
//   warp 0      TMA producer: A tile 128 x 128 B and two B tiles 128 x 128 B per
//               stage (4 stages of 48 KB), 128-byte swizzle;
//   warp 1      allocates the 512 TMEM columns and issues tcgen05.mma from one
//               lane (M=128, N=256, fp32 accumulate), commits to mbarriers;
//   warps 2..   epilogue: tcgen05.ld of the accumulator rows (one TMEM lane per
//               thread), activation / requantisation / scatter, global stores.
// bf16: two 256-column accumulators ping-pong between work items, so the
// epilogue of one item overlaps the main loop of the next.
// fp8: the block scales change every 128-deep K block, so the MMA writes each K
// block into one of two 256-column partial accumulators and eight epilogue
// warps add partial * (a_scale * w_scale) into fp32 registers while the MMA
// fills the other partial -- software promotion, since the scales are fp32.
//
// Work items are ordered expert by expert, then by N tile, then by M tile, so
// the M tiles of one expert that share a weight tile run side by side (the
// weight tile is read from HBM once) and an expert's activations stay in L2
// while its N tiles stream past.
//
// Every wait is bounded (see mbar_wait): a wait that gives up records
// MOE_ERR_TIMEOUT and the CTA unwinds, frees its TMEM and returns.
#include <cudaTypedefs.h>

#include <algorithm>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int BM = MOE_BLOCK_M;   // 128 rows per tile = TMEM lanes
constexpr int BN = 256;           // MMA N
constexpr int BKB = 128;          // bytes of K per stage (one 128-byte swizzle row)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BKB;             // 16 KB
constexpr int B_HALF_BYTES = 128 * BKB;       // 16 KB
constexpr int STAGE_BYTES = A_BYTES + 2 * B_HALF_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*barriers, exchange*/ + 1024 /*alignment*/ + 2048;

enum Kind { kGemm1 = 0, kGemm2 = 1 };

template <bool kFP8>
struct Cfg {
  static constexpr int kEpiWarps = kFP8 ? 8 : 4;
  static constexpr int kThreads = 64 + kEpiWarps * 32;
  static constexpr int kElemBytes = kFP8 ? 1 : 2;
  static constexpr int kBK = BKB / kElemBytes;  // K elements per stage
  static constexpr int kMmaK = kFP8 ? 32 : 16;  // K per tcgen05.mma
  static constexpr uint32_t kIdesc = make_idesc(kFP8 ? 0u : 1u, BM, BN);
};

struct GemmParams {
  const int32_t* offsets;      // [E + 1]
  const int32_t* tile_map;     // [num_tiles][2] (expert, first row)
  const int32_t* num_tiles;    // [1]
  const int32_t* sorted_slot;  // gemm2 scatter target rows; NULL = identity
  int K;                       // contraction depth (H for gemm1, I for gemm2)
  int NT;                      // N tiles per expert
  int I;                       // gemm1: h columns (the up half starts at row I of w13[e])
  int H;                       // gemm2: output columns
  int b_rows;                  // rows of one expert's weight matrix (2I or H)
  int s_pad;                   // row stride of the transposed scale arrays
  const float* a_scale_t;      // fp8: [K/128][s_pad] scales of the A rows
  const float* w_scale;        // fp8: [E][b_rows/128][K/128]
  void* out;                   // gemm1: h [rows][I]; gemm2: y [T*k][H] bf16
  float* out_scale_t;          // gemm1 fp8: [I/128][s_pad]
};

struct WorkItem {
  int e, row0, row_end, n;
};

__device__ __forceinline__ WorkItem decode(const GemmParams& p, int w) {
  WorkItem it;
  const int mt_base = w / p.NT;  // an M tile of the item's expert
  it.e = __ldg(p.tile_map + 2 * mt_base);
  const int r0 = __ldg(p.tile_map + 2 * mt_base + 1);
  const int off = __ldg(p.offsets + it.e);
  it.row_end = __ldg(p.offsets + it.e + 1);
  const int mstart = mt_base - (r0 - off) / BM;
  const int mcnt = (it.row_end - off + BM - 1) / BM;
  const int local = w - mstart * p.NT;
  it.n = local / mcnt;
  it.row0 = off + (local % mcnt) * BM;
  return it;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

template <bool kFP8, int kKind>
__global__ void __launch_bounds__(Cfg<kFP8>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmParams p) {
  using C = Cfg<kFP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // [2] accumulator ready
  uint64_t* tempty = tfull + 2;       // [2] accumulator drained
  uint64_t* xbar = tempty + 2;        // fp8 gemm1: row amax exchange between column halves
  uint64_t* drain = xbar + 1;         // teardown after a failed wait: MMA pipe drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* amax_x = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256);  // [2 items][2 halves][BM]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], C::kEpiWarps * 32);
    }
    mbar_init(xbar, C::kEpiWarps * 32);
    mbar_init(drain, 1);
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int total = __ldg(p.num_tiles) * p.NT;
  const int KB = p.K / C::kBK;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_a = policy_evict_last();
    const uint64_t pol_b = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    long long fills = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const WorkItem it = decode(p, w);
      int brow0, brow1;
      if (kKind == kGemm1) {
        brow0 = it.e * p.b_rows + it.n * 128;           // gate rows
        brow1 = it.e * p.b_rows + p.I + it.n * 128;     // up rows
      } else {
        brow0 = it.e * p.b_rows + it.n * 256;
        brow1 = brow0 + 128;
      }
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = warp_wait(&empty[stage], phase ^ 1))) break;
        if (lane == 0) {
          uint8_t* sA = smem + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          const int kx = kb * C::kBK;
          tma_load_2d(sA, &tmA, kx, it.row0, &full[stage], pol_a);
          tma_load_2d(sA + A_BYTES, &tmB, kx, brow0, &full[stage], pol_b);
          tma_load_2d(sA + A_BYTES + B_HALF_BYTES, &tmB, kx, brow1, &full[stage], pol_b);
        }
        __syncwarp();
        ++fills;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (status_failed() && lane == 0) {
      // wait (bounded) for the copies this CTA still has in flight: the last fill of each stage
      for (long long i = fills - 1; i >= 0 && i >= fills - STAGES; --i)
        mbar_wait(&full[i % STAGES], (uint32_t)((i / STAGES) & 1), false, 100000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      if (!kFP8) {
        if (!(ok = warp_wait(&tempty[acc], acc_phase ^ 1))) break;
        tc_fence_after();
      }
      for (int kb = 0; kb < KB; ++kb) {
        if (kFP8) {
          if (!(ok = warp_wait(&tempty[acc], acc_phase ^ 1))) break;
          tc_fence_after();
        }
        if (!(ok = warp_wait(&full[stage], phase))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b0 = a0 + A_BYTES;
          const uint32_t d = tmem + acc * BN;
#pragma unroll
          for (int kk = 0; kk < BKB / (C::kMmaK * C::kElemBytes); ++kk) {
            const uint32_t koff = kk * C::kMmaK * C::kElemBytes;
            const uint32_t accum = kFP8 ? (kk > 0) : (kb > 0 || kk > 0);
            if (kFP8)
              mma_fp8(d, sw128_desc(a0 + koff), sw128_desc(b0 + koff), C::kIdesc, accum);
            else
              mma_bf16(d, sw128_desc(a0 + koff), sw128_desc(b0 + koff), C::kIdesc, accum);
          }
          tc_commit(&empty[stage]);
          if (kFP8) tc_commit(&tfull[acc]);
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
        if (kFP8) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
      }
      if (!kFP8 && ok) {
        if (lane == 0) tc_commit(&tfull[acc]);
        __syncwarp();
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp - 2;
    const int quarter = warp & 3;      // TMEM lanes this warp may access
    const int half = q / 4;            // fp8: which half of the columns
    const int r = quarter * 32 + lane; // tile row == TMEM lane
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    int xbuf = 0;
    uint32_t xphase = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const WorkItem it = decode(p, w);
      const int prow = it.row0 + r;
      const bool valid = prow < it.row_end;
      if (!kFP8) {
        if (!(ok = warp_wait(&tfull[acc], acc_phase))) break;
        tc_fence_after();
        const uint32_t tb = tmem + lane_addr + acc * BN;
        if (kKind == kGemm1) {
          __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(p.out) + (size_t)prow * p.I + it.n * 128;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float g[32], u[32];
            tmem_ld32(tb + c * 32, g);
            tmem_ld32(tb + 128 + c * 32, u);
            tmem_ld_wait();
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(hrow + c * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 o;
                o.x = pack_bf16x2(silu_mul(g[8 * v + 0], u[8 * v + 0]), silu_mul(g[8 * v + 1], u[8 * v + 1]));
                o.y = pack_bf16x2(silu_mul(g[8 * v + 2], u[8 * v + 2]), silu_mul(g[8 * v + 3], u[8 * v + 3]));
                o.z = pack_bf16x2(silu_mul(g[8 * v + 4], u[8 * v + 4]), silu_mul(g[8 * v + 5], u[8 * v + 5]));
                o.w = pack_bf16x2(silu_mul(g[8 * v + 6], u[8 * v + 6]), silu_mul(g[8 * v + 7], u[8 * v + 7]));
                dst[v] = o;
              }
            }
          }
        } else {
          const int f = valid ? (p.sorted_slot ? __ldg(p.sorted_slot + prow) : prow) : 0;
          __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(p.out) + (size_t)f * p.H + it.n * 256;
          const int ncols = min(256, p.H - it.n * 256);
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            float v[32];
            tmem_ld32(tb + c * 32, v);
            tmem_ld_wait();
            if (valid && c * 32 < ncols) {
              uint4* dst = reinterpret_cast<uint4*>(yrow + c * 32);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint4 o;
                o.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
                o.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
                o.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
                o.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
                dst[j] = o;
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      } else {
        // fp8: promote every K block's partial into registers.
        // gemm1: this thread owns h columns [64 half, +64): gate TMEM columns
        //        [64 half, +64) and up columns [128 + 64 half, +64).
        // gemm2: this thread owns output columns [128 half, +128).
        float accv[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) accv[i] = 0.f;
        const int KBs = p.K / 128;
        const int nbw = p.b_rows / 128;
        const float* sw = p.w_scale + (size_t)it.e * nbw * KBs;
        int wb0, wb1;  // weight-scale block rows for column groups 0..63 / 64..127 of accv
        if (kKind == kGemm1) {
          wb0 = it.n;
          wb1 = p.I / 128 + it.n;
        } else {
          wb0 = wb1 = min(2 * it.n + half, nbw - 1);
        }
        const float* sa = p.a_scale_t + it.row0 + r;  // + kb * s_pad
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = warp_wait(&tfull[acc], acc_phase))) break;
          tc_fence_after();
          const float a_s = __ldg(sa + (size_t)kb * p.s_pad);
          const float s0 = a_s * __ldg(sw + (size_t)wb0 * KBs + kb);
          const float s1 = a_s * __ldg(sw + (size_t)wb1 * KBs + kb);
          const uint32_t tb = tmem + lane_addr + acc * BN;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            // gemm1: chunks 0,1 gate, 2,3 up; gemm2: 4 consecutive chunks
            const int col = kKind == kGemm1 ? (c < 2 ? 64 * half + 32 * c : 128 + 64 * half + 32 * (c - 2))
                                            : 128 * half + 32 * c;
            float v[32];
            tmem_ld32(tb + col, v);
            tmem_ld_wait();
            const float sc = (kKind == kGemm1 && c >= 2) ? s1 : s0;
#pragma unroll
            for (int i = 0; i < 32; ++i) accv[32 * c + i] = fmaf(v[i], sc, accv[32 * c + i]);
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
        if (!ok) break;
        if (kKind == kGemm1) {
          // h = silu(g) * u for 64 columns, then E4M3 G(128) over the 128 columns of this row
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            accv[i] = silu_mul(accv[i], accv[64 + i]);
            amax = fmaxf(amax, fabsf(accv[i]));
          }
          // exchange with the warp holding the other 64 columns of these rows (bounded wait)
          float* xb = amax_x + xbuf * 2 * BM;
          xb[half * BM + r] = amax;
          mbar_arrive(xbar);
          if (!(ok = warp_wait(xbar, xphase))) break;
          amax = fmaxf(amax, xb[(1 - half) * BM + r]);
          xphase ^= 1;
          xbuf ^= 1;
          const float s = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
          if (valid) {
            uint8_t* hrow = static_cast<uint8_t*>(p.out) + (size_t)prow * p.I + it.n * 128 + 64 * half;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t wds[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int i0 = 16 * v + 4 * j;
                const uint32_t lo = (uint32_t)__nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(accv[i0], s), __fdiv_rn(accv[i0 + 1], s)), __NV_SATFINITE, __NV_E4M3);
                const uint32_t hi = (uint32_t)__nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(accv[i0 + 2], s), __fdiv_rn(accv[i0 + 3], s)), __NV_SATFINITE, __NV_E4M3);
                wds[j] = lo | (hi << 16);
              }
              reinterpret_cast<uint4*>(hrow)[v] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
            }
            if (half == 0) p.out_scale_t[(size_t)it.n * p.s_pad + prow] = s;
          }
        } else {
          const int c0 = it.n * 256 + 128 * half;
          if (valid && c0 < p.H) {
            const int f = p.sorted_slot ? __ldg(p.sorted_slot + prow) : prow;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + (size_t)f * p.H + c0);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              uint4 o;
              o.x = pack_bf16x2(accv[8 * j + 0], accv[8 * j + 1]);
              o.y = pack_bf16x2(accv[8 * j + 2], accv[8 * j + 3]);
              o.z = pack_bf16x2(accv[8 * j + 4], accv[8 * j + 5]);
              o.w = pack_bf16x2(accv[8 * j + 6], accv[8 * j + 7]);
              dst[j] = o;
            }
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  // After a failed wait some MMAs may still be in flight: wait (bounded) for
  // the MMA pipe to drain before the TMEM is released.
  if (warp == 1 && status_failed()) {
    if (lane == 0) {
      tc_commit(drain);
      mbar_wait(drain, 0, false, 100000000ull);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// gather: one warp per sorted row p.  Copies the row of token sorted_slot[p]/k
// (unless codes are not wanted) and, for fp8, writes its scales transposed.
__global__ void __launch_bounds__(256)
    gather_kernel(const uint8_t* __restrict__ a1q, const float* __restrict__ a1q_scale,
                  const int32_t* __restrict__ sorted_slot, int S, int top_k, int row_bytes, int ngroups,
                  uint8_t* __restrict__ A, float* __restrict__ a_scale_t, int s_pad) {
  const int p = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (p >= S) return;
  const int t = sorted_slot ? __ldg(sorted_slot + p) / top_k : p;
  if (A) {
    const uint4* src = reinterpret_cast<const uint4*>(a1q + (size_t)t * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(A + (size_t)p * row_bytes);
    const int nv = row_bytes / 16;
    for (int i = lane; i < nv; i += 32) dst[i] = __ldg(src + i);
  }
  if (a_scale_t)
    for (int g = lane; g < ngroups; g += 32) a_scale_t[(size_t)g * s_pad + p] = __ldg(a1q_scale + (size_t)t * ngroups + g);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D K-major map over [rows][k] with a box of (128 bytes of K) x 128 rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, bool fp8, long long k, long long rows) {
  auto enc = get_encode();
  if (!enc) return false;
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(k * esz)};
  cuuint32_t box[2] = {(cuuint32_t)(BKB / esz), 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kFP8, int kKind>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, int grid, cudaStream_t s) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<kFP8, kKind>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  gemm_kernel<kFP8, kKind><<<grid, Cfg<kFP8>::kThreads, SMEM_BYTES, s>>>(a, b, p);
  return cudaGetLastError();
}

struct WsLayout {
  size_t A, As, h, hs, total;
  int s_pad;
};

inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(long long S, int H, int I, bool fp8) {
  WsLayout L;
  const int esz = fp8 ? 1 : 2;
  L.s_pad = (int)(((S + BM + 3) / 4) * 4);
  size_t off = 0;
  L.A = off;
  off = al256(off + (size_t)S * H * esz);
  L.As = off;
  off = al256(off + (fp8 ? (size_t)(H / 128) * L.s_pad * 4 : 0));
  L.h = off;
  off = al256(off + (size_t)S * I * esz);
  L.hs = off;
  off = al256(off + (fp8 ? (size_t)(I / 128) * L.s_pad * 4 : 0));
  L.total = off;
  return L;
}

}  // namespace

MOE_DEFINE_STATUS_READER(experts_status)

}  // namespace moe

using namespace moe;

extern "C" size_t moe_workspace_size(int T, int H, int I, int E, int top_k, const moe_quant_config* qc) {
  if (!qc || T < 0 || H <= 0 || I <= 0 || E < 1 || top_k < 1) return 0;
  return ws_layout((long long)T * top_k, H, I, qc->act == MOE_DT_FP8_E4M3).total;
}

extern "C" moe_status_t moe_experts(const void* a1q, const float* a1q_scale, const void* w13, const float* w13_scale,
                                    const void* w2, const float* w2_scale, const int32_t* expert_offsets,
                                    const int32_t* sorted_slot, const int32_t* tile_map, const int32_t* num_tiles,
                                    int T, int H, int I, int E, int top_k, const moe_quant_config* qc,
                                    void* fused_expert_output, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_ARG(qc && T >= 0 && H > 0 && I > 0 && E >= 1 && top_k >= 1 && top_k <= E);
  const bool fp8 = qc->act == MOE_DT_FP8_E4M3;
  if (fp8) {
    if (qc->act_group != 128 || qc->weight != MOE_DT_FP8_E4M3 || qc->w_block_n != 128 || qc->w_block_k != 128)
      return MOE_ERR_UNSUPPORTED;
  } else if (qc->act != MOE_DT_BF16 || qc->weight != MOE_DT_BF16) {
    return MOE_ERR_UNSUPPORTED;
  }
  MOE_CHECK_ARG(H % 128 == 0 && I % 128 == 0);
  const long long S = (long long)T * top_k;
  MOE_CHECK_ARG(fits_int32(S + 2 * BM) && fits_int32((long long)E * 2 * I) && fits_int32((long long)E * H));
  if (S == 0) return MOE_OK;
  MOE_CHECK_ARG(a1q && w13 && w2 && expert_offsets && tile_map && num_tiles && fused_expert_output);
  MOE_CHECK_ARG(sorted_slot || (E == 1 && top_k == 1));
  MOE_CHECK_ARG(!fp8 || (a1q_scale && w13_scale && w2_scale));
  MOE_CHECK_ARG(aligned16(a1q) && aligned16(w13) && aligned16(w2) && aligned16(fused_expert_output));
  const WsLayout L = ws_layout(S, H, I, fp8);
  if (!ws || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_CHECK_ARG(aligned16(ws));
  const int cap = moe_tile_map_capacity((int)S, E, BM);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const int esz = fp8 ? 1 : 2;
  const bool gather_rows = sorted_slot != nullptr;
  const void* A = gather_rows ? (const void*)(wsb + L.A) : a1q;
  float* As = fp8 ? reinterpret_cast<float*>(wsb + L.As) : nullptr;
  void* h = wsb + L.h;
  float* hs = fp8 ? reinterpret_cast<float*>(wsb + L.hs) : nullptr;

  if (gather_rows || fp8) {
    const unsigned grid = (unsigned)((S + 7) / 8);
    gather_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(a1q), a1q_scale, sorted_slot, (int)S, top_k,
                                       H * esz, H / 128, gather_rows ? wsb + L.A : nullptr, As, L.s_pad);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }

  CUtensorMap mA1, mB1, mA2, mB2;
  if (!make_map(&mA1, A, fp8, H, S) || !make_map(&mB1, w13, fp8, H, (long long)E * 2 * I) ||
      !make_map(&mA2, h, fp8, I, S) || !make_map(&mB2, w2, fp8, I, (long long)E * H))
    return MOE_ERR_CUDA;

  const int nsm = num_sms();
  GemmParams p1 = {};
  p1.offsets = expert_offsets;
  p1.tile_map = tile_map;
  p1.num_tiles = num_tiles;
  p1.sorted_slot = sorted_slot;
  p1.K = H;
  p1.NT = I / 128;
  p1.I = I;
  p1.H = H;
  p1.b_rows = 2 * I;
  p1.s_pad = L.s_pad;
  p1.a_scale_t = As;
  p1.w_scale = w13_scale;
  p1.out = h;
  p1.out_scale_t = hs;
  const int grid1 = (int)std::min<long long>(nsm, (long long)cap * p1.NT);

  GemmParams p2 = p1;
  p2.K = I;
  p2.NT = (H + 255) / 256;
  p2.b_rows = H;
  p2.a_scale_t = hs;
  p2.w_scale = w2_scale;
  p2.out = fused_expert_output;
  p2.out_scale_t = nullptr;
  const int grid2 = (int)std::min<long long>(nsm, (long long)cap * p2.NT);

  cudaError_t e;
  if (fp8) {
    e = launch_gemm<true, kGemm1>(mA1, mB1, p1, grid1, s);
    if (e == cudaSuccess) e = launch_gemm<true, kGemm2>(mA2, mB2, p2, grid2, s);
  } else {
    e = launch_gemm<false, kGemm1>(mA1, mB1, p1, grid1, s);
    if (e == cudaSuccess) e = launch_gemm<false, kGemm2>(mA2, mB2, p2, grid2, s);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
