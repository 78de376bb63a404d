// moe_experts: grouped expert MLPs on tcgen05 tensor cores.
//
// "Fused MoE Kernel Features" (vLLM design doc), section "Fused Experts
// Kernels": every expert runs two GEMMs with an activation between them
// (SiLU-and-mul, the SwiGLU default), consumes the prepared (possibly
// quantised) activations and writes its rows in the original activation type.
// For the fp8 G(128) format each token carries one scale per 128 channels and
// each weight one scale per 128x128 block.
//
// Launches on the caller's stream:
//   plan   : one block turns the 128-row tile map into the unit groups below and
//            clears the split-unit flags of both GEMMs
//   gather : a1q rows -> A rows in expert order (sorted_slot), fp8 scales
//            transposed to [K/128][rows], NVFP4 scale rows copied beside them;
//            skipped for the identity case
//   gemm1  : h = act(A w13_g^T, A w13_u^T), bf16, fp8 G(128) requantised, or bf16
//            then quantised by a separate pass ("A"/"T" fp8, NVFP4)
//   gemm2  : y[sorted_slot[p]] = h_p w2^T, bf16 rows scattered token-major
// moe_layer_fused runs the whole bf16 step (route to finalize) as one cooperative
// kernel whose GEMM phases are the same GEMM (gemm_body).
//
// GEMM design (one persistent CTA per SM):
//   unit   one weight tile (256 rows of w13 -- 128 gate + 128 up -- or of w2)
//          times a group of MG 128-row M tiles of one expert.  MG = 2 (bf16
//          only: when two-tile units of full tiles fill between half a wave and
//          one wave, as a deep-K gemm2's do) loads the weight tile once per K
//          step for both tiles; MG = 1 otherwise.  Units run expert by expert,
//          then N tile, then group.
//   warp 0 TMA producer: per stage one box of the MG A tiles and one box of
//          the 256 weight rows (gemm1: a 3-D box of the gate and the up block;
//          gemm2: 256 consecutive rows), 128-byte swizzle (MG = 2: 3 stages x
//          64 KB; MG = 1: 4 stages x 48 KB; NVFP4 adds the stage's 16-byte scale
//          rows of the A rows and the weight rows, 54 KB).  Two boxes per stage
//          rather than one per 128 rows: the copy engine moves about a third
//          more bytes per SM when its boxes are fewer and larger.
//   warp 1 allocates the 512 TMEM columns and issues tcgen05.mma from one lane
//          (M=128, N=256 per M tile, fp32 accumulate; kind::f16, kind::f8f6f4, or
//          the block-scaled kind::mxf4nvf4 for NVFP4).
//   epilogue warps (bf16 and NVFP4: 4, one per TMEM lane quarter; fp8: 8, two
//          per quarter): tcgen05.ld of accumulator rows (one TMEM lane per
//          thread).  bf16 MG = 1 ping-pongs two accumulators so one unit's
//          epilogue overlaps the next unit's main loop.  fp8: the block scales
//          change every 128-deep K block, so the MMA writes each K block into one
//          of two partial accumulators that the epilogue scales and adds into
//          fp32 registers (software promotion; the scales are fp32).  NVFP4: one
//          accumulator (the other half of the TMEM holds the stages' block
//          scales, which the epilogue warps copy there from shared memory before
//          the MMAs of the stage).
//   problems  one launch may carry two expert problems (moe_experts_multi: a
//          layer's routed experts and its shared expert): their units are
//          numbered one after the other and share the schedule below.
//   schedule  decode-sized problems (at most 16 slots per expert, K of 32+
//          blocks) with fewer units than half the CTAs split the (unit, K block)
//          iterations into equal contiguous ranges, one per CTA ("stream-K");
//          otherwise whole units go to the CTAs in the order the CTAs ask for
//          them (a launch-wide counter; round-robin when no counter is given),
//          so units that share a weight tile run side by side on neighbouring
//          SMs and a CTA that starts late takes fewer units.  A unit cut by a range
//          boundary is finished by the CTA holding its first K blocks: it waits
//          (bounded) for the later segments' fp32 partials and adds them in
//          segment order, so results do not depend on timing.  Those later
//          segments are always the first work of their CTAs and never wait, so
//          the waits cannot form a cycle while all CTAs are resident.
//
// Every wait is bounded: a wait that gives up records MOE_ERR_TIMEOUT and the
// CTA unwinds, drains its in-flight copies and MMAs, frees its TMEM and
// returns.
#include <cudaTypedefs.h>

#include <algorithm>

#include "moe_common.cuh"
#include "moe_route.cuh"

namespace moe {
namespace {

constexpr int BM = MOE_BLOCK_M;  // 128 rows per M tile = TMEM lanes
constexpr int BN = 256;          // MMA N
constexpr int BKB = 128;         // bytes of K per stage (one 128-byte swizzle row)
constexpr int A_BYTES = BM * BKB;        // 16 KB per M tile
constexpr int B_HALF_BYTES = 128 * BKB;  // 16 KB per 128 weight rows
constexpr int TMEM_COLS = 512;
// epilogue warps: bf16 4 (warps 2-5, one per TMEM lane quarter, all columns of its
// rows); fp8 8 (warps 4-11, two per lane quarter, half of the columns each: the
// promotion keeps 128 fp32 accumulators per thread).  The fp8 block is three full
// warpgroups -- warps 2 and 3 idle -- so that the registers can be moved between
// them (setmaxnreg): the producer and MMA warpgroup gives up most of its share and
// the epilogue warpgroups take it, enough to stage 64 accumulator columns per
// tensor-memory load beside the 128 promoted sums.
template <bool kFP8>
struct Warps {
  static constexpr int EPI = kFP8 ? 8 : 4;
  static constexpr int FIRST_EPI = kFP8 ? 4 : 2;
  static constexpr int THREADS = (FIRST_EPI + EPI) * 32;
  static constexpr int EPI_THREADS = EPI * 32;
};
// fp8 register split: launched at kLaunchRegs per thread (the most 384 threads can
// have), the first warpgroup drops to kLowRegs and the two epilogue warpgroups rise
// to kHighRegs.  The sum must equal what the block was launched with:
// 128 * kLowRegs + 256 * kHighRegs == 384 * kLaunchRegs (the host checks the
// kernel's register count before the first launch).
constexpr int kLaunchRegs = 168, kLowRegs = 40, kHighRegs = 232;
static_assert(128 * kLowRegs + 256 * kHighRegs == 384 * kLaunchRegs, "register split must balance");

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
// Units are split across CTAs (stream-K) only when there are fewer than half as
// many units as CTAs (decode-sized work); otherwise whole units are dealt
// round-robin, where a short tail costs less than the split's fixed costs.
constexpr int SPLIT_BELOW_UNITS_PER_CTA_X2 = 1;
// Dynamic schedule (GemmParams::unit_ctr set): the producer warp takes each next unit
// from a launch-wide counter and hands its index to the MMA and epilogue warps through
// a ring of UNIT_SLOTS entries in shared memory.
constexpr int UNIT_SLOTS = 4;

enum Kind { kGemm1 = 0, kGemm2 = 1 };

// kFP4: NVFP4 operands (packed E2M1 pairs, 256 K elements per 128-byte row) with
// their E4M3 block scales staged beside each stage's tiles: 128 A rows and 256
// weight rows of 16 scale bytes (one per 16 K elements) per stage.
constexpr int SFA_BYTES = BM * 16;
constexpr int SFB_BYTES = 2 * 128 * 16;
// tensor memory of the NVFP4 GEMMs: one accumulator (columns 0-255) and, per
// stage, the block scales of its 4 MMAs: 4 A columns and 8 weight columns each
// (the layout of mma_nvf4), from column 256 on
constexpr int SF_TMEM_BASE = 256;
constexpr int SF_TMEM_STAGE = 4 * 4 + 4 * 8;

// kDec: decode-sized problems (at most 32 rows per tile): a stage holds the first 32 rows of
// the A tile (a 32-row box; the MMA still reads 128 rows, the last 96 from the weight tile
// beside them, and their accumulator lanes are never read) and the 12 KB saved per stage buy
// more stages (bf16: six instead of four; NVFP4: five, whose 32-row A scale boxes leave the
// other 96 rows' scale words stale, for rows never read either), so each SM has more weight
// bytes in flight and spends less of its copy bandwidth on padding rows.
template <bool kFP8, int kMG, bool kFP4 = false, bool kDec = false>
struct Cfg {
  static constexpr int MG = kMG;  // M tiles per unit
  static constexpr int A_STAGE = kDec ? A_BYTES / 4 : A_BYTES;  // A bytes per M tile in a stage
  static constexpr int STAGES = kDec ? (kFP4 ? 5 : 6) : (kMG == 2 ? 3 : 4);
  static constexpr int SFA_LOAD = kDec ? SFA_BYTES / 4 : SFA_BYTES;  // NVFP4: A scale bytes copied per stage
  static constexpr int STAGE_BYTES = MG * A_STAGE + 2 * B_HALF_BYTES + (kFP4 ? SFA_BYTES + SFB_BYTES : 0);
  static constexpr int kBK = kFP4 ? 2 * BKB : (kFP8 ? BKB : BKB / 2);  // K elements per stage
  static constexpr int kMapK = kFP4 ? BKB : kBK;  // the same in units of the tensor maps' elements
  static constexpr int kMmaBytes = 32;            // bytes of K per tcgen05.mma (K = 16 bf16, 32 fp8, 64 fp4)
  static constexpr uint32_t kIdesc = kFP4 ? make_idesc_nvf4(BM, BN) : make_idesc(kFP8 ? 0u : 1u, BM, BN);
  static constexpr int PARTIAL_FLOATS = MG * BM * BN;  // one split-unit partial
  // fp8: ring of per-K-block scales (128 activation-row scales + 2 weight-block scales)
  static constexpr int SCALE_SLOTS = 8;
  static constexpr int SCALE_SLOT_FLOATS = 132;
  static constexpr int SCALE_RING_BYTES = kFP8 ? SCALE_SLOTS * SCALE_SLOT_FLOATS * 4 : 0;
  // fp8: per epilogue warp a 32-row x 32-column bf16 staging tile for the gemm2 output
  // (80-byte rows: conflict-free for the row-per-lane writes and the 8-rows-per-store reads)
  static constexpr int OUT_STAGE_STRIDE = 80;
  static constexpr int OUT_STAGE_BYTES = kFP8 ? Warps<kFP8>::EPI * 32 * OUT_STAGE_STRIDE : 0;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 4096 /*barriers, exchange*/ + SCALE_RING_BYTES +
                                    OUT_STAGE_BYTES +
                                    1024 /*align*/;
  static_assert(!kFP4 || (!kFP8 && kMG == 1), "NVFP4 units hold one M tile");
  static_assert(!kDec || (!kFP8 && kMG == 1), "decode stages: bf16 or NVFP4 units of one tile");
  static_assert(!kFP4 || SF_TMEM_BASE + STAGES * SF_TMEM_STAGE <= TMEM_COLS, "NVFP4 scales must fit the TMEM");
};

struct GemmParams {
  const int32_t* offsets;      // [E + 1] (batched format: expert e's slab starts at offsets[e])
  const int32_t* counts;       // batched format: [E] rows of each slab; NULL: rows end at offsets[e + 1]
  const int32_t* group_map;    // [groups][2] (expert, first row), built by plan_kernel
  const int32_t* num_groups;   // [1]
  const int32_t* sorted_slot;  // gemm2 scatter target rows; NULL = identity
  int K;                       // contraction depth (H for gemm1, I for gemm2)
  int NT;                      // N tiles per expert
  int I;                       // gemm1: h columns (the up half starts at row I of w13[e])
  int H;                       // gemm2: output columns
  int b_rows;                  // rows of one expert's weight matrix (2I or H)
  int s_pad;                   // row stride of the transposed scale arrays
  int a_kstride;               // fp8: stride of a_scale_t between K blocks (0: one scale per row)
  const float* a_scale_t;      // fp8: [K/128][a_kstride] scales of the A rows
  const float* w_scale;        // fp8: [E][b_rows/128][K/128]
  const float* a_gscale;       // NVFP4: [1] global scale of the A rows
  const float* w_gscale;       // NVFP4: [E] global scale of each expert's weights
  void* out;                   // gemm1: h [rows][I]; gemm2: y [T*k][H] bf16
  float* out_scale_t;          // gemm1 fp8: [I/128][s_pad]
  int allow_split;             // decode-sized problem: few units may be split across CTAs (bf16 only)
  int* flags;                  // [units] arrivals on split units (zeroed by plan_kernel)
  float* partials;             // [gridDim.x][PARTIAL_FLOATS] one split-segment partial per CTA
  int* unit_ctr;               // problem 0: launch-wide unit counter (zeroed before the launch) for the
                               // dynamic schedule; NULL: the static schedule (Sched)
};

// Up to two expert problems in one launch (moe_experts_multi: typically a layer's
// routed experts and its shared expert).  Their units are numbered one after the
// other, problem 0 first, and share the schedule, the K depth and the per-CTA
// split partials.
constexpr int kMaxProblems = 2;
struct GemmProblems {
  GemmParams p[kMaxProblems];
  int nprob;
};

struct Unit {
  int e, row0, row_end, n;  // rows [row0, row_end) of expert e (at most MG*BM), N tile n
};

// Loads of the schedule's tables (offsets, group map, unit count, sorted slots).
// kCoh: the tables were written earlier in the same kernel (the single-launch
// layer), so they are read coherently (ld.global.cg); otherwise an earlier launch
// wrote them and the read-only path (ld.global.nc) is used.
template <bool kCoh>
__device__ __forceinline__ int ld_tab(const int32_t* p) {
  return kCoh ? __ldcg(p) : __ldg(p);
}

template <int MG, bool kCoh>
__device__ __forceinline__ Unit decode(const GemmParams& p, int u) {
  Unit it;
  const int gb = u / p.NT;  // a group of the unit's expert
  it.e = ld_tab<kCoh>(p.group_map + 2 * gb);
  const int r0 = ld_tab<kCoh>(p.group_map + 2 * gb + 1);
  const int off = ld_tab<kCoh>(p.offsets + it.e);
  const int end = p.counts ? off + ld_tab<kCoh>(p.counts + it.e) : ld_tab<kCoh>(p.offsets + it.e + 1);
  const int gstart = gb - (r0 - off) / (MG * BM);
  const int gcnt = (end - off + MG * BM - 1) / (MG * BM);
  const int local = u - gstart * p.NT;
  it.n = local / gcnt;
  it.row0 = off + (local % gcnt) * (MG * BM);
  it.row_end = min(it.row0 + MG * BM, end);
  return it;
}

// The segments (unit, K blocks [kb0, kb1)) one CTA processes, in order.
struct Sched {
  bool rr;
  int U, KB, G, c;
  long long i, i1, total;
  int u_next;
  __device__ void init(int units, int kb, int grid, int cta, bool allow_split) {
    U = units;
    KB = kb;
    c = cta;
    total = (long long)units * kb;
    rr = !allow_split || 2 * units >= SPLIT_BELOW_UNITS_PER_CTA_X2 * grid;
    // stream-K uses at most one CTA per iteration, so that no range is empty
    G = rr ? grid : (int)std::min<long long>(grid, std::max<long long>(total, 1));
    u_next = cta;
    if (rr || cta < G) {
      i = total * cta / G;
      i1 = total * (cta + 1) / G;
    } else {
      i = i1 = 0;
    }
  }
  __device__ bool next(int& u, int& kb0, int& kb1) {
    if (rr) {
      if (u_next >= U) return false;
      u = u_next;
      kb0 = 0;
      kb1 = KB;
      u_next += G;
      return true;
    }
    if (i >= i1) return false;
    u = (int)(i / KB);
    kb0 = (int)(i % KB);
    kb1 = (int)std::min<long long>(KB, kb0 + (i1 - i));
    i += kb1 - kb0;
    return true;
  }
  // CTA whose range holds iteration `it` (stream-K mode)
  __device__ int cta_of(long long it) const { return (int)(((it + 1) * G - 1) / total); }
};

// Bounded wait of a whole warp on the phase with parity `parity`: every lane tests
// it (the test itself suspends the warp for a while); between tests the warp sleeps
// briefly, leaving issue slots and shared-memory cycles to the warps that keep the
// pipeline fed (measured: 2-3 % on the fp8 GEMMs, 0.5-1 % on the bf16 ones).  Gives
// up, false, when a failure is recorded or after the wait limit (recording
// MOE_ERR_TIMEOUT).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    __nanosleep(64);
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    if (status_failed()) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      if ((threadIdx.x & 31) == 0) record_timeout();
      return false;
    }
  }
}


// Epilogue threads of the CTA that finishes a split unit: one thread polls the
// unit's arrival count (the other threads polling the same L2 line would
// crowd it), then releases the rest through a shared-memory barrier.  A CTA
// finishes at most one split unit per launch (its last segment), so the
// barrier's phase is always 0.  Bounded: false after a timeout.
__device__ __forceinline__ bool wait_split_partials(const int* flag, int target, uint64_t* fixbar) {
  if ((threadIdx.x >> 5) == Warps<false>::FIRST_EPI) {  // (split units are bf16 or NVFP4)
    // the whole first epilogue warp polls in step (one lane loads, a shuffle shares
    // the value): a lone polling lane would be starved by its warp-mates' waits
    const int lane = threadIdx.x & 31;
    const uint64_t t0 = global_ns();
    while (true) {
      int v = 0;
      if (lane == 0) asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
      v = __shfl_sync(0xffffffffu, v, 0);
      if (v >= target) break;
      if (status_failed()) break;
      if (global_ns() - t0 > kWaitLimitNs) {
        if (lane == 0) record_timeout();
        break;
      }
      __nanosleep(100);
    }
    if (lane == 0) mbar_arrive(fixbar);  // on failure the status word is set; release the others anyway
  }
  const bool ok = mbar_wait(fixbar, 0);
  return __all_sync(0xffffffffu, ok && !status_failed());
}

// A later segment's partial is written: every lane fences its own stores, then
// one atomic per warp counts the warp's 32 threads.
__device__ __forceinline__ void signal_split_partial(int* flag) {
  __threadfence();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) atomicAdd(flag, 32);
}

// Activations between the two GEMMs (moe_activation_t): act_gate is the gate's
// function alone (the *_NO_MUL forms), act_mul the gated form h(g, u).  The
// sigmoids divide with the fast fp32 division intrinsic (a couple of fp32 ulps,
// far below the bf16 rounding of h; for a denominator past 2^126, i.e. g below
// about -87, it returns 0, the value h has in bf16 there): the IEEE division took
// most of an NVFP4 GEMM1 epilogue, which the next unit's MMAs wait for.
__device__ __forceinline__ float act_silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }
__device__ __forceinline__ float act_gelu(float g) { return 0.5f * g * (1.0f + erff(g * 0.70710678118654752f)); }
__device__ __forceinline__ float act_gelu_tanh(float g) {
  return 0.5f * g * (1.0f + tanhf(0.79788456080286536f * (g + 0.044715f * g * g * g)));
}
template <int kAct>
__device__ __forceinline__ float act_gate(float g) {
  if (kAct == MOE_ACT_GELU || kAct == MOE_ACT_GELU_NO_MUL) return act_gelu(g);
  if (kAct == MOE_ACT_GELU_TANH) return act_gelu_tanh(g);
  return act_silu(g);
}
template <int kAct>
__device__ __forceinline__ float act_mul(float g, float u) {
  if (kAct == MOE_ACT_SWIGLUOAI) {
    // gpt-oss SwiGLU: gate clamped above at 7, up clamped to [-7, 7], sigmoid(1.702 g)
    const float gc = fminf(g, 7.0f), uc = fminf(fmaxf(u, -7.0f), 7.0f);
    return (uc + 1.0f) * __fdividef(gc, 1.0f + __expf(-1.702f * gc));
  }
  return act_gate<kAct>(g) * u;
}

// The persistent GEMM (see the top of the file), run by every CTA of the grid over the
// dynamic shared memory `smem_raw`.  `standalone`: the CTA's only work (it gives up its
// TMEM allocation permit after allocating); otherwise one phase of a longer kernel,
// which may allocate again and re-initialise the barriers, so they are invalidated at
// the end.
template <bool kFP8, int kKind, int kMG, int kAct, bool kHB16, bool kFP4, bool kCoh = false, bool kDec = false>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tmA, const CUtensorMap& tmA2, const CUtensorMap& tmB,
                                          const CUtensorMap& tmA_1, const CUtensorMap& tmA2_1,
                                          const CUtensorMap& tmB_1, const CUtensorMap& tmSA,
                                          const CUtensorMap& tmSB, const GemmProblems& pp, uint8_t* smem_raw,
                                          bool standalone) {
  using C = Cfg<kFP8, kMG, kFP4, kDec>;
  // gemm1 forms: a gated activation reads 128 gate + 128 up rows per unit (one 3-D
  // box); a *_NO_MUL one reads 256 consecutive gate rows, like gemm2
  constexpr bool kNoMul = kKind == kGemm1 && (kAct == MOE_ACT_SILU_NO_MUL || kAct == MOE_ACT_GELU_NO_MUL);
  constexpr bool kPair = kKind == kGemm1 && !kNoMul;
  constexpr int EPI_WARPS = Warps<kFP8>::EPI;
  constexpr int EPI_THREADS = Warps<kFP8>::EPI_THREADS;
  constexpr int MG = C::MG;
  constexpr int STAGES = C::STAGES;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ctrl = smem + STAGES * C::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // [2] accumulator ready
  uint64_t* tempty = tfull + 2;      // [2] accumulator drained
  uint64_t* xbar = tempty + 2;       // fp8 gemm1: row amax exchange between column halves
  uint64_t* drain = xbar + 1;        // teardown after a failed wait
  uint64_t* fixbar = drain + 1;      // stream-K: the later segments' partials of this CTA's split unit are in
  uint64_t* sfull = fixbar + 1;      // fp8 scale ring: [SCALE_SLOTS] slot filled
  uint64_t* sempty = sfull + C::SCALE_SLOTS;  // [SCALE_SLOTS] slot read by every epilogue warp
  uint64_t* ufull = sempty + C::SCALE_SLOTS;  // dynamic schedule: [UNIT_SLOTS] unit index written
  uint64_t* uempty = ufull + UNIT_SLOTS;      // [UNIT_SLOTS] unit index read by the MMA and epilogue warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(uempty + UNIT_SLOTS);
  volatile int* unit_ring = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [UNIT_SLOTS]
  float* scale_ring = reinterpret_cast<float*>(ctrl + 4096);  // fp8: [SCALE_SLOTS][SCALE_SLOT_FLOATS]
  uint8_t* out_stage = ctrl + 4096 + C::SCALE_RING_BYTES;  // fp8 gemm2: [EPI warps][32][OUT_STAGE_STRIDE]
  float* amax_x = reinterpret_cast<float*>(ctrl + 512);  // [2 items][2 halves][BM]
  // control block: barriers, TMEM address and unit ring below byte 512, the amax exchange up
  // to 2560, the NVFP4 scale barriers from 3072, the fp8 scale ring from 4096
  static_assert((2 * STAGES + 4 + 3 + 2 * C::SCALE_SLOTS + 2 * UNIT_SLOTS) * 8 + 4 + 4 * UNIT_SLOTS <= 512,
                "control block overlaps the amax exchange");
  static_assert(512 + 2 * 2 * BM * 4 <= 3072 && 3072 + STAGES * 8 <= 4096, "control block layout");
  uint64_t* sfready = reinterpret_cast<uint64_t*>(ctrl + 3072);  // NVFP4: [STAGES] stage's scales in TMEM
  // bf16 split units: the finished rows (own accumulator + later segments' partials),
  // [BM][FIX_STRIDE] fp32 over the stage buffers
  constexpr int FIX_STRIDE = 257;  // odd stride: row-per-thread writes hit distinct banks
  static_assert(BM * FIX_STRIDE * 4 <= STAGES * C::STAGE_BYTES, "fix-up sums must fit the stages");
  float* fix = reinterpret_cast<float*>(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], EPI_WARPS);  // one arrival per epilogue warp
    }
    mbar_init(xbar, EPI_WARPS);
    if (kFP4)
      for (int st = 0; st < STAGES; ++st) mbar_init(&sfready[st], EPI_WARPS);
    mbar_init(drain, 1);
    mbar_init(fixbar, 1);
    for (int i = 0; i < C::SCALE_SLOTS; ++i) {
      mbar_init(&sfull[i], 32);  // one cp.async arrival per producer lane
      mbar_init(&sempty[i], EPI_WARPS);
    }
    for (int i = 0; i < UNIT_SLOTS; ++i) {
      mbar_init(&ufull[i], 1);
      mbar_init(&uempty[i], 1 + EPI_WARPS);
    }
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    if (MG == 2) prefetch_tensormap(&tmA2);
    prefetch_tensormap(&tmB);
    if (kFP4) {
      prefetch_tensormap(&tmSA);
      prefetch_tensormap(&tmSB);
    }
    if (pp.nprob > 1) {
      prefetch_tensormap(&tmA_1);
      if (MG == 2) prefetch_tensormap(&tmA2_1);
      prefetch_tensormap(&tmB_1);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    if (standalone) tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const GemmParams& p0 = pp.p[0];
  const int units0 = ld_tab<kCoh>(p0.num_groups) * p0.NT;  // problem 1's units follow problem 0's
  const int units = units0 + (pp.nprob > 1 ? ld_tab<kCoh>(pp.p[1].num_groups) * pp.p[1].NT : 0);
  const int KB = p0.K / C::kBK;
  Sched sched;
  // fp8 units are never split: its register promotion leaves no room for the split logic
  constexpr bool kSplit = !kFP8;
  // (split units have one M tile: the fix-up below sums one tile's rows)
  sched.init(units, KB, gridDim.x, blockIdx.x, kSplit && MG == 1 && p0.allow_split);
  int u, kb0, kb1;
  // The dynamic schedule hands whole units to CTAs in the order they ask, so a CTA that
  // starts late (its SM still held by another kernel) takes fewer of them instead of
  // finishing late.  Units that share a weight tile are taken at about the same time by
  // neighbouring askers, as in the static schedule.
  // (units split across CTAs keep the static ranges: their fix-up needs to know which CTA
  // holds which segment)
  const bool dyn = p0.unit_ctr != nullptr && sched.rr;
  long long useq = 0;  // units taken through the ring by this warp
  auto next_unit_producer = [&]() -> bool {
    if (!dyn) return sched.next(u, kb0, kb1);
    const int slot = (int)(useq % UNIT_SLOTS);
    if (!warp_wait(&uempty[slot], (uint32_t)(((useq / UNIT_SLOTS) & 1) ^ 1))) return false;
    int v = 0;
    if (lane == 0) {
      v = atomicAdd(p0.unit_ctr, 1);
      if (v >= units) v = -1;  // no unit left: tells the other warps to stop
      unit_ring[slot] = v;
      mbar_arrive(&ufull[slot]);
    }
    u = __shfl_sync(0xffffffffu, v, 0);
    ++useq;
    kb0 = 0;
    kb1 = KB;
    return u >= 0;
  };
  auto next_unit_consumer = [&]() -> bool {
    if (!dyn) return sched.next(u, kb0, kb1);
    const int slot = (int)(useq % UNIT_SLOTS);
    if (!warp_wait(&ufull[slot], (uint32_t)((useq / UNIT_SLOTS) & 1))) return false;
    u = unit_ring[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&uempty[slot]);
    ++useq;
    kb0 = 0;
    kb1 = KB;
    return u >= 0;
  };

  if (warp < Warps<kFP8>::FIRST_EPI) {
  // fp8: this warpgroup (producer, MMA issuer, two idle warps) hands registers to the
  // epilogue warpgroups, which take them at the top of their branch
  if (kFP8) setmaxnreg_dec<kLowRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_a = policy_evict_last();
    const uint64_t pol_b = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    long long fills = 0;
    bool ok = true;
    while (ok && next_unit_producer()) {
      const int prob = u >= units0;
      const GemmParams& p = pp.p[prob];
      const CUtensorMap* mA = prob ? &tmA_1 : &tmA;
      const CUtensorMap* mA2 = prob ? &tmA2_1 : &tmA2;
      const CUtensorMap* mB = prob ? &tmB_1 : &tmB;
      const Unit it = decode<MG, kCoh>(p, u - (prob ? units0 : 0));
      const int mcnt = (it.row_end - it.row0 + BM - 1) / BM;
      // gemm1: gate block n of expert e and the up block I rows further (3-D map
      // [2E][I][K], z = 2e gate, 2e + 1 up); gemm2: w2 rows [256 n, +256) of expert e
      const int brow = kPair ? it.n * 128 : it.e * p.b_rows + it.n * 256;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!(ok = warp_wait(&empty[stage], phase ^ 1))) break;
        if (kFP8) {
          // this K block's scales into the ring, copied asynchronously by all lanes:
          // the activation scales of the tile's 128 rows and the two weight-block scales
          const int slot = (int)(fills % C::SCALE_SLOTS);
          if (!(ok = warp_wait(&sempty[slot], (uint32_t)(((fills / C::SCALE_SLOTS) & 1) ^ 1)))) break;
          float* dst = scale_ring + slot * C::SCALE_SLOT_FLOATS;
          const float* asrc = p.a_scale_t + (size_t)kb * p.a_kstride + it.row0;
#pragma unroll
          for (int j = 0; j < 4; ++j) cp_async_4(dst + lane * 4 + j, asrc + lane * 4 + j);
          if (lane == 0) {
            const int KBs = p.K / 128, nbw = p.b_rows / 128;
            const float* sw = p.w_scale + (size_t)it.e * nbw * KBs;
            const int wb0 = kPair ? it.n : min(2 * it.n, nbw - 1);
            const int wb1 = kPair ? p.I / 128 + it.n : min(2 * it.n + 1, nbw - 1);
            cp_async_4(dst + 128, sw + (size_t)wb0 * KBs + kb);
            cp_async_4(dst + 129, sw + (size_t)wb1 * KBs + kb);
          }
          cp_async_arrive(&sfull[slot]);
        }
        if (lane == 0) {
          uint8_t* sA = smem + stage * C::STAGE_BYTES;
          uint8_t* sB = sA + MG * C::A_STAGE;
          mbar_arrive_expect_tx(&full[stage],
                                mcnt * C::A_STAGE + 2 * B_HALF_BYTES + (kFP4 ? C::SFA_LOAD + SFB_BYTES : 0));
          const int kx = kb * C::kMapK;
          if (kFP4) {
            // the block scales of the stage: 16 bytes of each A row and of each weight row
            uint8_t* sSF = sB + 2 * B_HALF_BYTES;
            tma_load_2d(sSF, &tmSA, kb * 16, it.row0, &full[stage], pol_a);
            if (kPair)
              tma_load_3d(sSF + SFA_BYTES, &tmSB, kb * 16, brow, 2 * it.e, &full[stage], pol_b);
            else
              tma_load_2d(sSF + SFA_BYTES, &tmSB, kb * 16, brow, &full[stage], pol_b);
          }
          if (MG == 2 && mcnt == 2)
            tma_load_2d(sA, mA2, kx, it.row0, &full[stage], pol_a);  // both M tiles, one 256-row box
          else
            tma_load_2d(sA, mA, kx, it.row0, &full[stage], pol_a);
          if (kPair)
            tma_load_3d(sB, mB, kx, brow, 2 * it.e, &full[stage], pol_b);
          else
            tma_load_2d(sB, mB, kx, brow, &full[stage], pol_b);
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
      // wait (bounded) for the copies still in flight: the last fill of each stage
      for (long long i = fills - 1; i >= 0 && i >= fills - STAGES; --i)
        mbar_wait(&full[i % STAGES], (uint32_t)((i / STAGES) & 1), false, 100000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    // fp8: ping-pong partial per K block; bf16 MG=1: ping-pong accumulator per
    // unit; bf16 MG=2: one accumulator set of MG tiles
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    while (ok && next_unit_consumer()) {
      const int prob = u >= units0;
      const Unit it = decode<MG, kCoh>(pp.p[prob], u - (prob ? units0 : 0));
      const int mcnt = (it.row_end - it.row0 + BM - 1) / BM;
      if (!kFP8) {
        if (!(ok = warp_wait(&tempty[acc], acc_phase ^ 1))) break;
        tc_fence_after();
      }
      for (int kb = kb0; kb < kb1; ++kb) {
        if (kFP8) {
          if (!(ok = warp_wait(&tempty[acc], acc_phase ^ 1))) break;
          tc_fence_after();
        }
        if (!(ok = warp_wait(&full[stage], phase))) break;
        if (kFP4 && !(ok = warp_wait(&sfready[stage], phase))) break;  // the stage's scales are in TMEM
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b0 = a0 + MG * C::A_STAGE;
          for (int m = 0; m < mcnt; ++m) {
            const uint32_t d = tmem + ((kFP8 || MG == 1) ? acc * BN : m * BN);
#pragma unroll
            for (int kk = 0; kk < BKB / C::kMmaBytes; ++kk) {
              const uint32_t koff = kk * C::kMmaBytes;
              const uint32_t accum = kFP8 ? (kk > 0) : (kb > kb0 || kk > 0);
              if (kFP4) {
                const uint32_t sf = tmem + SF_TMEM_BASE + stage * SF_TMEM_STAGE;
                mma_nvf4(d, sw128_desc(a0 + koff), sw128_desc(b0 + koff), C::kIdesc, sf + 4 * kk, sf + 16 + 8 * kk,
                         accum);
              } else if (kFP8)
                mma_fp8(d, sw128_desc(a0 + m * C::A_STAGE + koff), sw128_desc(b0 + koff), C::kIdesc, accum);
              else
                mma_bf16(d, sw128_desc(a0 + m * C::A_STAGE + koff), sw128_desc(b0 + koff), C::kIdesc, accum);
            }
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
        if (MG == 1 && !kFP4) acc ^= 1;  // (NVFP4: one accumulator, the scales take the other half)
        if (acc == 0) acc_phase ^= 1;
      }
    }
  }
  } else {
    // ------------------------------------------------------------ epilogue
    if (kFP8) setmaxnreg_inc<kHighRegs>();
    const int q = warp - Warps<kFP8>::FIRST_EPI;
    const int quarter = warp & 3;        // TMEM lanes this warp may access
    const int sub = q / 4;               // fp8: column half (bf16: always 0)
    const int r = quarter * 32 + lane;   // row within an M tile == TMEM lane
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    float* my_partial = p0.partials + (size_t)blockIdx.x * C::PARTIAL_FLOATS;  // [MG][BM][BN] (bf16 splits)
    int acc = 0;
    uint32_t acc_phase = 0;
    int xbuf = 0;
    uint32_t xphase = 0;
    long long sfill = 0;  // fp8: K blocks consumed from the scale ring
    int fstage = 0;       // NVFP4: stages whose scales this warp has put in TMEM
    uint32_t fphase = 0;
    bool ok = true;
    while (ok && next_unit_consumer()) {
      const int prob = u >= units0;
      const GemmParams& p = pp.p[prob];
      const int lu = u - (prob ? units0 : 0);  // the unit within its problem (split flags)
      const Unit it = decode<MG, kCoh>(p, lu);
      const int prow = it.row0 + r;  // row of the first M tile (fp8: the only one)
      const bool valid = prow < it.row_end;
      // split-unit role: 0 whole, 1 first segment (finishes the unit), 2 later segment
      const int role = !kSplit ? 0 : (kb0 == 0 && kb1 == KB) ? 0 : (kb0 == 0 ? 1 : 2);
      int c_first = 0, c_last = -1;
      if (role == 1) {
        c_first = blockIdx.x + 1;
        c_last = sched.cta_of((long long)u * KB + KB - 1);
      }
      // thread-private slot of a split-unit partial (bf16): 256 columns of (M tile m, row r)
      // at poff + m * BM * 256
      const size_t poff = (size_t)r * 256;
      // NVFP4: the accumulators hold sums of (E2M1 x block scale) products; the two
      // operands' global scales multiply the finished sums
      const float alpha = kFP4 ? __ldg(p.a_gscale) * __ldg(p.w_gscale + it.e) : 1.0f;
      if (kFP4) {
        // Before the unit's epilogue, every K block's block scales go from the stage
        // into tensor memory in the layout mma_nvf4 reads; each warp writes the same
        // copy into its own lane quarter: lane l holds the scale words of A rows
        // l + 32 c (columns 4 kk + c of the stage's slot, kk the MMA) and of weight
        // rows 128 hh + l + 32 c (columns 16 + 8 kk + 4 hh + c).
        bool fed = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!(fed = warp_wait(&full[fstage], fphase))) break;
          const uint8_t* sSF = smem + fstage * C::STAGE_BYTES + MG * C::A_STAGE + 2 * B_HALF_BYTES;
          uint4 ra[4], rb[8];
#pragma unroll
          for (int c = 0; c < 4; ++c) ra[c] = *reinterpret_cast<const uint4*>(sSF + (lane + 32 * c) * 16);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            rb[c] = *reinterpret_cast<const uint4*>(sSF + SFA_BYTES + (128 * (c >> 2) + lane + 32 * (c & 3)) * 16);
          uint32_t va[16], vb[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            va[c] = ra[c].x;
            va[4 + c] = ra[c].y;
            va[8 + c] = ra[c].z;
            va[12 + c] = ra[c].w;
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            vb[c] = rb[c].x;
            vb[8 + c] = rb[c].y;
            vb[16 + c] = rb[c].z;
            vb[24 + c] = rb[c].w;
          }
          const uint32_t col = tmem + lane_addr + SF_TMEM_BASE + fstage * SF_TMEM_STAGE;
          tmem_st16(col, va);
          tmem_st32(col + 16, vb);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sfready[fstage]);
          if (++fstage == STAGES) {
            fstage = 0;
            fphase ^= 1;
          }
        }
        if (!(ok = fed)) break;
      }

      if (!kFP8) {
        // one warp per TMEM lane quarter: rows r of each M tile of the group, 8 chunks of
        // 32 columns (gemm1: chunks 0-3 gate, 4-7 up)
        if (!(ok = warp_wait(&tfull[acc], acc_phase))) break;
        tc_fence_after();
        if (role == 1) {
          // The first segment of a split unit finishes it, column-parallel over all
          // epilogue threads (decode-sized units have few valid rows, which a
          // row-per-thread epilogue would leave to one thread): its own accumulator rows
          // go to shared memory (the stage buffers are free: this segment is the CTA's
          // last work and its MMAs are complete), the later segments' partials are added
          // in segment order, every load independent, then the outputs are written.
          // Split units have one M tile.  Every epilogue warp arrives at both barrier
          // phases, whatever its status, so that none waits in vain.
          ok = wait_split_partials(p.flags + lu, (c_last - c_first + 1) * EPI_THREADS, fixbar);
          const int nrows = min(BM, it.row_end - it.row0);
          const int tid = threadIdx.x - 64;
          const uint32_t tb = tmem + lane_addr + acc * BN;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            float v[32];
            tmem_ld32(tb + c * 32, v);
            tmem_ld_wait();
            if (r < nrows) {
#pragma unroll
              for (int j = 0; j < 32; ++j) fix[r * FIX_STRIDE + c * 32 + j] = v[j];
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(xbar);
          ok = warp_wait(xbar, 0) && ok;
          const int n = nrows * 256;
          if (ok) {
            for (int i0 = tid; i0 < n; i0 += 4 * EPI_THREADS) {
              float a[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int i = i0 + k * EPI_THREADS;
                a[k] = i < n ? fix[(i >> 8) * FIX_STRIDE + (i & 255)] : 0.f;
              }
#pragma unroll 4
              for (int cc = c_first; cc <= c_last; ++cc) {
                const float* src = p.partials + (size_t)cc * C::PARTIAL_FLOATS;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  if (i0 + k * EPI_THREADS < n) a[k] += __ldcg(src + i0 + k * EPI_THREADS);
              }
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int i = i0 + k * EPI_THREADS;
                if (i < n) fix[(i >> 8) * FIX_STRIDE + (i & 255)] = a[k] * alpha;
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(xbar);
          ok = warp_wait(xbar, 1) && ok;
          if (ok) {
            if (kPair) {
              // h[row][128 n + col] = act(gate, up), two columns per thread and step
              __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out) + it.n * 128;
              for (int i = tid; i < nrows * 64; i += EPI_THREADS) {
                const int row = i >> 6, col = 2 * (i & 63);
                const float* f = fix + row * FIX_STRIDE + col;
                const uint32_t o = pack_bf16x2(act_mul<kAct>(f[0], f[128]), act_mul<kAct>(f[1], f[129]));
                *reinterpret_cast<uint32_t*>(h + (size_t)(it.row0 + row) * p.I + col) = o;
              }
            } else if (kNoMul) {
              // h[row][256 n + col] = act(gate)
              __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out) + it.n * 256;
              const int ncols = min(256, p.I - it.n * 256);
              for (int i = tid; i < nrows * 128; i += EPI_THREADS) {
                const int row = i >> 7, col = 2 * (i & 127);
                if (col >= ncols) continue;
                const float* f = fix + row * FIX_STRIDE + col;
                *reinterpret_cast<uint32_t*>(h + (size_t)(it.row0 + row) * p.I + col) =
                    pack_bf16x2(act_gate<kAct>(f[0]), act_gate<kAct>(f[1]));
              }
            } else {
              // y[sorted_slot[row]][256 n + col], two columns per thread and step
              const int ncols = min(256, p.H - it.n * 256);
              for (int i = tid; i < nrows * 128; i += EPI_THREADS) {
                const int row = i >> 7, col = 2 * (i & 127);
                if (col >= ncols) continue;
                const int mrow = it.row0 + row;
                const int f = p.sorted_slot ? ld_tab<kCoh>(p.sorted_slot + mrow) : mrow;
                const float* x = fix + row * FIX_STRIDE + col;
                *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.out) + (size_t)f * p.H + it.n * 256 + col) =
                    pack_bf16x2(x[0], x[1]);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
          if (MG == 1 && !kFP4) acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
          continue;
        }
        const int mcnt = (it.row_end - it.row0 + BM - 1) / BM;
        for (int m = 0; m < mcnt; ++m) {
          const int mrow = prow + m * BM;
          const bool mvalid = mrow < it.row_end;
          const size_t mpoff = poff + (size_t)m * BM * 256;
          const uint32_t tb = tmem + lane_addr + (MG == 2 ? m * BN : acc * BN);
          if (role == 2) {
            // later segment: park the fp32 partial for the CTA that finishes the unit
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              float v[32];
              tmem_ld32(tb + c * 32, v);
              tmem_ld_wait();
              if (mvalid) {
                float4* dst = reinterpret_cast<float4*>(my_partial + mpoff + c * 32);
#pragma unroll
                for (int j = 0; j < 8; ++j) __stcg(dst + j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
              }
            }
          } else if (kPair) {
            __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(p.out) + (size_t)mrow * p.I + it.n * 128;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              float g[32], uu[32];
              tmem_ld32(tb + c * 32, g);
              tmem_ld32(tb + 128 + c * 32, uu);
              tmem_ld_wait();
              if (kFP4) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  g[j] *= alpha;
                  uu[j] *= alpha;
                }
              }
              if (mvalid) {
                uint4* dst = reinterpret_cast<uint4*>(hrow + c * 32);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  uint4 o;
                  o.x = pack_bf16x2(act_mul<kAct>(g[8 * v + 0], uu[8 * v + 0]), act_mul<kAct>(g[8 * v + 1], uu[8 * v + 1]));
                  o.y = pack_bf16x2(act_mul<kAct>(g[8 * v + 2], uu[8 * v + 2]), act_mul<kAct>(g[8 * v + 3], uu[8 * v + 3]));
                  o.z = pack_bf16x2(act_mul<kAct>(g[8 * v + 4], uu[8 * v + 4]), act_mul<kAct>(g[8 * v + 5], uu[8 * v + 5]));
                  o.w = pack_bf16x2(act_mul<kAct>(g[8 * v + 6], uu[8 * v + 6]), act_mul<kAct>(g[8 * v + 7], uu[8 * v + 7]));
                  dst[v] = o;
                }
              }
            }
          } else if (kNoMul) {
            __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(p.out) + (size_t)mrow * p.I + it.n * 256;
            const int ncols = min(256, p.I - it.n * 256);
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              float v[32];
              tmem_ld32(tb + c * 32, v);
              tmem_ld_wait();
              if (kFP4) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= alpha;
              }
              if (mvalid && c * 32 < ncols) {
                uint4* dst = reinterpret_cast<uint4*>(hrow + c * 32);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint4 o;
                  o.x = pack_bf16x2(act_gate<kAct>(v[8 * j + 0]), act_gate<kAct>(v[8 * j + 1]));
                  o.y = pack_bf16x2(act_gate<kAct>(v[8 * j + 2]), act_gate<kAct>(v[8 * j + 3]));
                  o.z = pack_bf16x2(act_gate<kAct>(v[8 * j + 4]), act_gate<kAct>(v[8 * j + 5]));
                  o.w = pack_bf16x2(act_gate<kAct>(v[8 * j + 6]), act_gate<kAct>(v[8 * j + 7]));
                  dst[j] = o;
                }
              }
            }
          } else {
            const int f = mvalid ? (p.sorted_slot ? ld_tab<kCoh>(p.sorted_slot + mrow) : mrow) : 0;
            __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(p.out) + (size_t)f * p.H + it.n * 256;
            const int ncols = min(256, p.H - it.n * 256);
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              float v[32];
              tmem_ld32(tb + c * 32, v);
              tmem_ld_wait();
              if (kFP4) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= alpha;
              }
              if (mvalid && c * 32 < ncols) {
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
        }
        if (role == 2) signal_split_partial(p.flags + lu);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        if (MG == 1 && !kFP4) acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      } else {
        // fp8: promote every K block's partial into registers.
        // gemm1: this thread owns h columns [64 half, +64): gate TMEM columns
        //        [64 half, +64) and up columns [128 + 64 half, +64).
        // gemm2: this thread owns output columns [128 half, +128).
        const int half = sub;
        // gemm2: the slot this row's output goes to, loaded now so that its latency
        // passes under the K loop instead of stalling the unit's end
        const int f_out = kKind == kGemm2 && valid ? (p.sorted_slot ? ld_tab<kCoh>(p.sorted_slot + prow) : prow) : -1;
        // sums as pairs of columns: one packed two-wide fp32 FMA (each lane an IEEE fma)
        // per pair and K block
        float2 acc2[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc2[i] = make_float2(0.f, 0.f);
        for (int kb = kb0; kb < kb1; ++kb) {
          // scales of this K block from the ring the producer fills ahead of time
          const int slot = (int)(sfill % C::SCALE_SLOTS);
          if (!(ok = warp_wait(&sfull[slot], (uint32_t)((sfill / C::SCALE_SLOTS) & 1)))) break;
          const float* ring = scale_ring + slot * C::SCALE_SLOT_FLOATS;
          const float a_s = ring[r];
          // gemm1: accv[0..63] gate block, accv[64..127] up block; gemm2: this half's block
          const float s0 = a_s * ring[kPair ? 128 : 128 + half];
          const float s1 = a_s * ring[kPair ? 129 : 128 + half];
          __syncwarp();
          if (lane == 0) mbar_arrive(&sempty[slot]);
          ++sfill;
          if (!(ok = warp_wait(&tfull[acc], acc_phase))) break;
          tc_fence_after();
          const uint32_t tb = tmem + lane_addr + acc * BN;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            // two loads of 64 columns: gemm1 the gate block, then the up block; gemm2
            // two consecutive chunks
            const int col = kPair ? (c == 0 ? 64 * half : 128 + 64 * half) : 128 * half + 64 * c;
            float v[64];
            tmem_ld64_wait(tb + col, v);
            const float sc = (kPair && c == 1) ? s1 : s0;
            const float2 sc2 = make_float2(sc, sc);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              acc2[32 * c + i] = __ffma2_rn(make_float2(v[2 * i], v[2 * i + 1]), sc2, acc2[32 * c + i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
        if (!ok) break;
        float accv[128];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          accv[2 * i] = acc2[i].x;
          accv[2 * i + 1] = acc2[i].y;
        }
        // (fp8 units are never split: no partials to park or to add)
        if (kHB16) {
          // the "A"/"T" formats: h goes out in bf16 ([rows][I]); a later pass quantises it
          const int hc0 = kNoMul ? (2 * it.n + half) * 128 : it.n * 128 + 64 * half;
          const int nh = kNoMul ? 128 : 64;
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i < nh) accv[i] = kNoMul ? act_gate<kAct>(accv[i]) : act_mul<kAct>(accv[i], accv[64 + i]);
          if (valid && hc0 < p.I) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + (size_t)prow * p.I + hc0);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (8 * j >= nh) break;
              uint4 o;
              o.x = pack_bf16x2(accv[8 * j + 0], accv[8 * j + 1]);
              o.y = pack_bf16x2(accv[8 * j + 2], accv[8 * j + 3]);
              o.z = pack_bf16x2(accv[8 * j + 4], accv[8 * j + 5]);
              o.w = pack_bf16x2(accv[8 * j + 6], accv[8 * j + 7]);
              dst[j] = o;
            }
          }
        } else if (kNoMul) {
          // h = act(g) for this thread's 128 columns, which are one G(128) group (2n + half)
          const int grp = 2 * it.n + half;
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            accv[i] = act_gate<kAct>(accv[i]);
            amax = fmaxf(amax, fabsf(accv[i]));
          }
          const float s = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
          const float rs = __frcp_rn(s);
          if (valid && grp * 128 < p.I) {
            uint8_t* hrow = static_cast<uint8_t*>(p.out) + (size_t)prow * p.I + grp * 128;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              uint32_t wds[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int i0 = 16 * v + 4 * j;
                const uint32_t lo = (uint32_t)__nv_cvt_float2_to_fp8x2(
                    make_float2(div_rn_by(accv[i0], s, rs), div_rn_by(accv[i0 + 1], s, rs)), __NV_SATFINITE,
                    __NV_E4M3);
                const uint32_t hi = (uint32_t)__nv_cvt_float2_to_fp8x2(
                    make_float2(div_rn_by(accv[i0 + 2], s, rs), div_rn_by(accv[i0 + 3], s, rs)), __NV_SATFINITE,
                    __NV_E4M3);
                wds[j] = lo | (hi << 16);
              }
              reinterpret_cast<uint4*>(hrow)[v] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
            }
            p.out_scale_t[(size_t)grp * p.s_pad + prow] = s;
          }
        } else if (kPair) {
          // h = act(g, u) for 64 columns, then E4M3 G(128) over the 128 columns of this row
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            accv[i] = act_mul<kAct>(accv[i], accv[64 + i]);
            amax = fmaxf(amax, fabsf(accv[i]));
          }
          // exchange with the warp holding the other 64 columns of these rows (bounded wait)
          float* xb = amax_x + xbuf * 2 * BM;
          xb[half * BM + r] = amax;
          __syncwarp();
          if (lane == 0) mbar_arrive(xbar);
          if (!(ok = warp_wait(xbar, xphase))) break;
          amax = fmaxf(amax, xb[(1 - half) * BM + r]);
          xphase ^= 1;
          xbuf ^= 1;
          const float s = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
          const float rs = __frcp_rn(s);
          if (valid) {
            uint8_t* hrow = static_cast<uint8_t*>(p.out) + (size_t)prow * p.I + it.n * 128 + 64 * half;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t wds[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int i0 = 16 * v + 4 * j;
                const uint32_t lo = (uint32_t)__nv_cvt_float2_to_fp8x2(
                    make_float2(div_rn_by(accv[i0], s, rs), div_rn_by(accv[i0 + 1], s, rs)), __NV_SATFINITE,
                    __NV_E4M3);
                const uint32_t hi = (uint32_t)__nv_cvt_float2_to_fp8x2(
                    make_float2(div_rn_by(accv[i0 + 2], s, rs), div_rn_by(accv[i0 + 3], s, rs)), __NV_SATFINITE,
                    __NV_E4M3);
                wds[j] = lo | (hi << 16);
              }
              reinterpret_cast<uint4*>(hrow)[v] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
            }
            if (half == 0) p.out_scale_t[(size_t)it.n * p.s_pad + prow] = s;
          }
        } else {
          // y rows (scattered to their slots): a lane holds one row's 128 columns, so the
          // warp passes them through its staging tile 32 columns at a time and each store
          // then writes 64 contiguous bytes of each of 8 rows, not 16 bytes of 32 rows
          const int c0 = it.n * 256 + 128 * half;
          if (c0 < p.H) {  // (warp-uniform)
            const int f = f_out;
            uint8_t* stg = out_stage + (warp - Warps<kFP8>::FIRST_EPI) * 32 * C::OUT_STAGE_STRIDE;
            __nv_bfloat16* ybase = static_cast<__nv_bfloat16*>(p.out) + c0;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              uint4* srow = reinterpret_cast<uint4*>(stg + lane * C::OUT_STAGE_STRIDE);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int j = 32 * ch + 8 * q;
                uint4 o;
                o.x = pack_bf16x2(accv[j + 0], accv[j + 1]);
                o.y = pack_bf16x2(accv[j + 2], accv[j + 3]);
                o.z = pack_bf16x2(accv[j + 4], accv[j + 5]);
                o.w = pack_bf16x2(accv[j + 6], accv[j + 7]);
                srow[q] = o;
              }
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int rr = 8 * i + (lane & 7), pc = lane >> 3;  // row of the tile, 16-byte piece
                const int fr = __shfl_sync(0xffffffffu, f, rr);
                const uint4 v = *reinterpret_cast<const uint4*>(stg + rr * C::OUT_STAGE_STRIDE + pc * 16);
                if (fr >= 0) *reinterpret_cast<uint4*>(ybase + (size_t)fr * p.H + 32 * ch + 8 * pc) = v;
              }
              __syncwarp();
            }
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  // The MMA pipe drains (bounded wait) before the TMEM is released and the CTA exits:
  // after a failed wait MMAs may still be in flight, and on a normal exit the last
  // stages' commit arrivals on their empty barriers may still be pending -- once the CTA
  // has exited, its shared memory can belong to another CTA (a phase of a longer kernel
  // reuses its barriers too).
  if (warp == 1) {
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
  if (!standalone && threadIdx.x == 0) {
    // every barrier of this phase is idle: free them for the next phase's initialisation
    for (int s = 0; s < STAGES; ++s) {
      mbar_inval(&full[s]);
      mbar_inval(&empty[s]);
      if (kFP4) mbar_inval(&sfready[s]);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_inval(&tfull[a]);
      mbar_inval(&tempty[a]);
    }
    mbar_inval(xbar);
    mbar_inval(drain);
    mbar_inval(fixbar);
    for (int i = 0; i < C::SCALE_SLOTS; ++i) {
      mbar_inval(&sfull[i]);
      mbar_inval(&sempty[i]);
    }
    for (int i = 0; i < UNIT_SLOTS; ++i) {
      mbar_inval(&ufull[i]);
      mbar_inval(&uempty[i]);
    }
  }
}

template <bool kFP8, int kKind, int kMG, int kAct, bool kHB16, bool kFP4, bool kDec>
__global__ void __launch_bounds__(Warps<kFP8>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA_1,
                const __grid_constant__ CUtensorMap tmA2_1, const __grid_constant__ CUtensorMap tmB_1,
                const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                const __grid_constant__ GemmProblems pp) {
  extern __shared__ uint8_t smem_raw[];
  gemm_body<kFP8, kKind, kMG, kAct, kHB16, kFP4, false, kDec>(tmA, tmA2, tmB, tmA_1, tmA2_1, tmB_1, tmSA, tmSB, pp,
                                                              smem_raw, true);
}

// Groups of MG tiles of one expert (expert, first row) and their count, from
// the 128-row tile map.  Called by all threads of a 1024-thread block.
__device__ void build_groups(const int32_t* __restrict__ tile_map, int n, const int32_t* __restrict__ offsets, int MG,
                             int32_t* __restrict__ group_map, int32_t* __restrict__ num_groups) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n; base += 1024) {
    const int mt = base + threadIdx.x;
    int e = 0, r0 = 0, start = 0;
    if (mt < n) {
      e = tile_map[2 * mt];
      r0 = tile_map[2 * mt + 1];
      start = ((r0 - offsets[e]) / BM) % MG == 0;
    }
    int x = start;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const int w = warp_tot[lane];
      int wx = w;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wx, off);
        if (lane >= off) wx += y;
      }
      warp_tot[lane] = wx - w;
    }
    __syncthreads();
    const int idx = carry + warp_tot[warp] + x - start;
    if (start) {
      group_map[2 * idx] = e;
      group_map[2 * idx + 1] = r0;
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry = idx + start;
    __syncthreads();
  }
  if (threadIdx.x == 0) *num_groups = carry;
  __syncthreads();
}

// plan: the two-tile group maps of the GEMMs that use them and cleared split-unit
// flags (of every problem of the call).  One block.
__global__ void __launch_bounds__(1024)
    plan_kernel(const int32_t* __restrict__ tile_map, const int32_t* __restrict__ num_tiles,
                const int32_t* __restrict__ offsets, int mg1, int mg2, int32_t* __restrict__ gmap1,
                int32_t* __restrict__ ngroups1, int32_t* __restrict__ gmap2, int32_t* __restrict__ ngroups2,
                int* __restrict__ flags, int nflags) {
  const int n = *num_tiles;
  // (a GEMM of one-tile units reads the tile map itself)
  if (mg1 == 2) build_groups(tile_map, n, offsets, mg1, gmap1, ngroups1);
  if (mg2 == 2) build_groups(tile_map, n, offsets, mg2, gmap2, ngroups2);
  for (int i = threadIdx.x; i < nflags; i += 1024) flags[i] = 0;
}

// gather: one warp per sorted row p.  Copies the row of token sorted_slot[p]/k
// (unless codes are not wanted) and, for fp8, writes its scales transposed; for
// NVFP4 it also copies the row's block-scale bytes (sf_bytes of a1q_sf) to ASF.
__global__ void __launch_bounds__(256)
    gather_kernel(const uint8_t* __restrict__ a1q, const float* __restrict__ a1q_scale,
                  const int32_t* __restrict__ sorted_slot, int S, int top_k, int row_bytes, int ngroups,
                  uint8_t* __restrict__ A, float* __restrict__ a_scale_t, int s_pad, int scale_stride,
                  int* __restrict__ flags, int nflags, const uint8_t* __restrict__ a1q_sf, int sf_bytes,
                  uint8_t* __restrict__ ASF) {
  // (when no plan launch runs, the gather also clears the split-unit flags)
  for (int i = blockIdx.x * 256 + threadIdx.x; i < nflags; i += gridDim.x * 256) flags[i] = 0;
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
    for (int g = lane; g < ngroups; g += 32)
      a_scale_t[(size_t)g * s_pad + p] = __ldg(a1q_scale + (size_t)t * scale_stride + g);
  if (ASF) {
    const uint4* src = reinterpret_cast<const uint4*>(a1q_sf + (size_t)t * sf_bytes);
    uint4* dst = reinterpret_cast<uint4*>(ASF + (size_t)p * sf_bytes);
    for (int i = lane; i < sf_bytes / 16; i += 32) dst[i] = __ldg(src + i);
  }
}

// NVFP4 quantiser of bf16 rows [rows][C] (one thread per 16-element group, see
// nvfp4_group16), with the global scale at g: packed codes q [rows][C/2] and
// scale codes sf [rows][C/16].  rows = *nrows when nrows is given (the experts'
// intermediate: expert_offsets[E]), else max_rows.  weights (the prepare step's
// weight on the input, top-k 1): each row is first multiplied by bf16(weights[row])
// and rounded to bf16.
__global__ void __launch_bounds__(256)
    nvfp4_quant_kernel(const __nv_bfloat16* __restrict__ x, int C, long long max_rows,
                       const int32_t* __restrict__ nrows, const float* __restrict__ weights,
                       const float* __restrict__ g, uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;  // group index
  const int gpr = C / 16;
  const long long rows = nrows ? (long long)__ldg(nrows) : max_rows;
  if (i >= rows * gpr) return;
  const long long row = i / gpr;
  float v[16];
  float a[8];
  load_bf16x8(x + i * 16, a);
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = a[j];
  load_bf16x8(x + i * 16 + 8, a);
#pragma unroll
  for (int j = 0; j < 8; ++j) v[8 + j] = a[j];
  if (weights) {
    const float w = __bfloat162float(__float2bfloat16_rn(__ldg(weights + row)));
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __bfloat162float(__float2bfloat16_rn(v[j] * w));
  }
  uint8_t code;
  const uint64_t packed = nvfp4_group16(v, __ldg(g), code);
  reinterpret_cast<uint2*>(q)[i] = make_uint2((uint32_t)packed, (uint32_t)(packed >> 32));
  sf[i] = code;
}

// The "A" and "T" formats' intermediate: h rows [rows][I] in bf16 (rows =
// expert_offsets[E]) -> E4M3 codes hq and one scale per row hs (for "T" the
// tensor's scale repeated on every row, the layout gemm2 reads).
__global__ void __launch_bounds__(256)
    hquant_token_kernel(const __nv_bfloat16* __restrict__ hb, int I, const int32_t* __restrict__ offsets, int E,
                        uint8_t* __restrict__ hq, float* __restrict__ hs) {
  const int p = blockIdx.x;
  if (p >= __ldg(offsets + E)) return;  // block-uniform: the whole block leaves
  const int nv = I / 8;
  const __nv_bfloat16* row = hb + (size_t)p * I;
  float a = 0.f;
  for (int v = threadIdx.x; v < nv; v += 256) {
    float x[8];
    load_bf16x8(row + (size_t)v * 8, x);
    a = fmaxf(a, amax8(x));
  }
  const float sc = __fdiv_rn(fmaxf(block_amax<256>(a), 1e-10f), 448.0f);
  uint2* out = reinterpret_cast<uint2*>(hq + (size_t)p * I);
  for (int v = threadIdx.x; v < nv; v += 256) {
    float x[8];
    load_bf16x8(row + (size_t)v * 8, x);
    out[v] = e4m3x8(x, sc);
  }
  if (threadIdx.x == 0) hs[p] = sc;
}

__global__ void __launch_bounds__(256)
    hquant_tensor_amax_kernel(const __nv_bfloat16* __restrict__ hb, int I, const int32_t* __restrict__ offsets,
                              int E, unsigned* __restrict__ amax_bits) {
  const long long nvec = (long long)__ldg(offsets + E) * (I / 8);
  float a = 0.f;
  for (long long v = (long long)blockIdx.x * 256 + threadIdx.x; v < nvec; v += (long long)gridDim.x * 256) {
    float x[8];
    load_bf16x8(hb + v * 8, x);
    a = fmaxf(a, amax8(x));
  }
  a = block_amax<256>(a);
  if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(a));
}

__global__ void __launch_bounds__(256)
    hquant_tensor_kernel(const __nv_bfloat16* __restrict__ hb, int I, const int32_t* __restrict__ offsets, int E,
                         const unsigned* __restrict__ amax_bits, uint8_t* __restrict__ hq, float* __restrict__ hs) {
  const long long v = (long long)blockIdx.x * 256 + threadIdx.x;
  const int vpr = I / 8;
  if (v >= (long long)__ldg(offsets + E) * vpr) return;
  const float sc = __fdiv_rn(fmaxf(__uint_as_float(*amax_bits), 1e-10f), 448.0f);
  float x[8];
  load_bf16x8(hb + v * 8, x);
  reinterpret_cast<uint2*>(hq)[v] = e4m3x8(x, sc);
  if (v % vpr == 0) hs[v / vpr] = sc;
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

// 2-D K-major map over [rows][k] with a box of (128 bytes of K) x box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, bool fp8, long long k, long long rows, int box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(k * esz)};
  cuuint32_t box[2] = {(cuuint32_t)(BKB / esz), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// w13 [E][2I][k] viewed as [2E][I][k] (z = 2e: gate block, 2e + 1: up block of
// expert e); a box of (128 bytes of K) x 128 rows x 2 brings a gate block and
// its up block in one copy, the up rows 16 KB after the gate rows.
bool make_map_gate_up(CUtensorMap* m, const void* base, bool fp8, long long k, long long I, long long E) {
  auto enc = get_encode();
  if (!enc) return false;
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)k, (cuuint64_t)I, (cuuint64_t)(2 * E)};
  cuuint64_t strides[2] = {(cuuint64_t)(k * esz), (cuuint64_t)(I * k * esz)};
  cuuint32_t box[3] = {(cuuint32_t)(BKB / esz), 128, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Block-scale rows of an NVFP4 operand: 2-D map over [rows][row_bytes] bytes with a
// box of 16 bytes (one stage's 256 K elements) x box_rows rows, no swizzle.
bool make_map_sf(CUtensorMap* m, const void* base, long long row_bytes, long long rows, int box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {16, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The gate/up block-scale rows of w13 viewed as [2E][I][row_bytes] (the scale
// counterpart of make_map_gate_up): a box of 16 bytes x 128 rows x 2.
bool make_map_sf_gate_up(CUtensorMap* m, const void* base, long long row_bytes, long long I, long long E) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)row_bytes, (cuuint64_t)I, (cuuint64_t)(2 * E)};
  cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)(I * row_bytes)};
  cuuint32_t box[3] = {16, 128, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of one problem for one GEMM: A with one-tile and two-tile boxes,
// weights; NVFP4: the block-scale rows of A and of the weights.
struct GemmMaps {
  CUtensorMap a, a2, b, sa, sb;
};

template <bool kFP8, int kKind, int kMG, int kAct, bool kHB16 = false, bool kFP4 = false, bool kDec = false>
cudaError_t launch_gemm(const GemmMaps* m, const GemmProblems& pp, int grid, cudaStream_t s) {
  using C = Cfg<kFP8, kMG, kFP4, kDec>;
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<kFP8, kKind, kMG, kAct, kHB16, kFP4, kDec>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (kFP8) {
      // the fp8 kernel moves registers between its warpgroups (setmaxnreg): the split
      // balances only when the block launches with kLaunchRegs per thread; with fewer
      // the epilogue's increase could never be granted, so such a build never launches
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, gemm_kernel<kFP8, kKind, kMG, kAct, kHB16, kFP4, kDec>);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    }
    configured[dev] = 1;
  }
  const GemmMaps& m1 = pp.nprob > 1 ? m[1] : m[0];
  gemm_kernel<kFP8, kKind, kMG, kAct, kHB16, kFP4, kDec><<<grid, Warps<kFP8>::THREADS, C::SMEM_BYTES, s>>>(
      m[0].a, m[0].a2, m[0].b, m1.a, m1.a2, m1.b, m[0].sa, m[0].sb, pp);
  return cudaGetLastError();
}

// gemm1 with the activation chosen at run time (kHB16: fp8 mainloop, bf16 h out)
template <bool kFP8, int kMG, bool kHB16 = false, bool kFP4 = false, bool kDec = false>
cudaError_t launch_gemm1(int act, const GemmMaps* m, const GemmProblems& pp, int grid, cudaStream_t s) {
  switch (act) {
    case MOE_ACT_SILU: return launch_gemm<kFP8, kGemm1, kMG, MOE_ACT_SILU, kHB16, kFP4, kDec>(m, pp, grid, s);
    case MOE_ACT_GELU: return launch_gemm<kFP8, kGemm1, kMG, MOE_ACT_GELU, kHB16, kFP4, kDec>(m, pp, grid, s);
    case MOE_ACT_GELU_TANH:
      return launch_gemm<kFP8, kGemm1, kMG, MOE_ACT_GELU_TANH, kHB16, kFP4, kDec>(m, pp, grid, s);
    case MOE_ACT_SWIGLUOAI:
      return launch_gemm<kFP8, kGemm1, kMG, MOE_ACT_SWIGLUOAI, kHB16, kFP4, kDec>(m, pp, grid, s);
    case MOE_ACT_SILU_NO_MUL:
      return launch_gemm<kFP8, kGemm1, kMG, MOE_ACT_SILU_NO_MUL, kHB16, kFP4, kDec>(m, pp, grid, s);
    case MOE_ACT_GELU_NO_MUL:
      return launch_gemm<kFP8, kGemm1, kMG, MOE_ACT_GELU_NO_MUL, kHB16, kFP4, kDec>(m, pp, grid, s);
  }
  return cudaErrorInvalidValue;
}

inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of one call: per problem its gathered rows, transposed scales,
// intermediate and group maps; then the split flags of every problem and GEMM,
// contiguous so that one plan launch clears them; then one split partial per CTA.
struct ProbLayout {
  size_t A, As, h, hs, hb, hamax, gmap, ngroups, gmap2, ngroups2, flags1, flags2;
  int s_pad, nflags1, nflags2;
};
struct WsLayout {
  ProbLayout p[kMaxProblems];
  size_t flags, ctrs, partials, total;  // ctrs: the two GEMMs' unit counters, right after the flags
  int nflags;
};

// group: the fp8 activation format (128, MOE_GROUP_TOKEN or MOE_GROUP_TENSOR); the
// "A"/"T" formats add the bf16 intermediate and the tensor format's amax word.
WsLayout ws_layout(const moe_experts_problem* pr, int n, int H, bool fp8, int grid, int group,
                   bool rows_in_place = false) {
  WsLayout L{};
  const int esz = fp8 ? 1 : 2;
  const int MG = fp8 ? 1 : 2;  // the larger bound of either GEMM
  size_t off = 0;
  L.nflags = 0;
  for (int i = 0; i < n; ++i) {
    ProbLayout& P = L.p[i];
    const long long S = (long long)pr[i].T * pr[i].top_k;
    const int I = pr[i].I, E = pr[i].E;
    P.s_pad = (int)(((S + MG * BM + 3) / 4) * 4);
    const int cap_groups = std::max(1, moe_tile_map_capacity((int)S, E, BM));  // a group holds at least one tile
    P.nflags1 = cap_groups * (I / 128);
    P.nflags2 = cap_groups * ((H + 255) / 256);
    L.nflags += P.nflags1 + P.nflags2;
    P.A = off;
    off = al256(off + (rows_in_place ? 0 : (size_t)S * H * esz));
    P.As = off;
    off = al256(off + (fp8 ? (size_t)(H / 128) * P.s_pad * 4 : 0));
    P.h = off;
    off = al256(off + (size_t)S * I * esz);
    P.hs = off;
    off = al256(off + (fp8 ? (size_t)(I / 128) * P.s_pad * 4 : 0));
    const bool hb16 = fp8 && group != 128;
    P.hb = off;
    off = al256(off + (hb16 ? (size_t)S * I * 2 : 0));
    P.hamax = off;
    off = al256(off + (hb16 ? 4 : 0));
    P.gmap = off;
    off = al256(off + (size_t)cap_groups * 2 * 4);
    P.ngroups = off;
    off = al256(off + 4);
    P.gmap2 = off;
    off = al256(off + (size_t)cap_groups * 2 * 4);
    P.ngroups2 = off;
    off = al256(off + 4);
  }
  L.flags = off;
  size_t f = off;
  for (int i = 0; i < n; ++i) {
    L.p[i].flags1 = f;
    f += (size_t)L.p[i].nflags1 * 4;
    L.p[i].flags2 = f;
    f += (size_t)L.p[i].nflags2 * 4;
  }
  L.ctrs = f;  // contiguous with the flags: one clearing pass covers both
  f += 2 * 4;
  off = al256(f);
  L.partials = off;
  off = al256(off + (size_t)grid * MG * BM * BN * 4);
  L.total = off;
  return L;
}

// Grid of the persistent GEMMs: one CTA per SM (the workspace holds one
// split-unit partial per CTA, so its size depends on this).
int gemm_grid() { return num_sms(); }

bool quant_ok(const moe_quant_config* qc) {
  if (qc->act == MOE_DT_FP8_E4M3)
    return (qc->act_group == 128 || qc->act_group == MOE_GROUP_TOKEN || qc->act_group == MOE_GROUP_TENSOR) &&
           qc->weight == MOE_DT_FP8_E4M3 && qc->w_block_n == 128 && qc->w_block_k == 128;
  return qc->act == MOE_DT_BF16 && qc->weight == MOE_DT_BF16;
}

// The experts of one or more problems in the same launches.
moe_status_t experts_run(const moe_experts_problem* probs, int nprob, int H, const moe_quant_config* qc,
                         int activation, void* ws, size_t ws_bytes, cudaStream_t s) {
  MOE_CHECK_ARG(qc && probs && nprob >= 1 && nprob <= kMaxProblems && H > 0);
  if (activation < MOE_ACT_SILU || activation > MOE_ACT_GELU_NO_MUL || !quant_ok(qc)) return MOE_ERR_UNSUPPORTED;
  const bool no_mul = activation == MOE_ACT_SILU_NO_MUL || activation == MOE_ACT_GELU_NO_MUL;
  const bool fp8 = qc->act == MOE_DT_FP8_E4M3;
  const int group = qc->act_group;
  const bool hb16 = fp8 && group != 128;  // "A"/"T": bf16 h, then quantised per row or per tensor
  MOE_CHECK_ARG(H % 128 == 0 && fits_int32((long long)H * 8));
  // the problems with rows; several share the launches only in bf16 and with one K depth per GEMM
  moe_experts_problem pr[kMaxProblems];
  int n = 0;
  for (int i = 0; i < nprob; ++i) {
    const moe_experts_problem& q = probs[i];
    MOE_CHECK_ARG(q.T >= 0 && q.I > 0 && q.I % 128 == 0 && q.E >= 1 && q.top_k >= 1 && q.top_k <= q.E);
    const long long S = (long long)q.T * q.top_k;
    MOE_CHECK_ARG(fits_int32(S + 4 * BM) && fits_int32((long long)q.E * 2 * q.I) && fits_int32((long long)q.E * H));
    if (S == 0) continue;
    MOE_CHECK_ARG(q.a1q && q.w13 && q.w2 && q.expert_offsets && q.tile_map && q.num_tiles && q.fused_expert_output);
    MOE_CHECK_ARG(q.sorted_slot || (q.E == 1 && q.top_k == 1));
    MOE_CHECK_ARG(!fp8 || (q.a1q_scale && q.w13_scale && q.w2_scale));
    MOE_CHECK_ARG(aligned16(q.a1q) && aligned16(q.w13) && aligned16(q.w2) && aligned16(q.fused_expert_output));
    pr[n++] = q;
  }
  if (n == 0) return MOE_OK;
  if (n > 1 && (fp8 || pr[0].I != pr[1].I)) return MOE_ERR_UNSUPPORTED;
  const int grid = gemm_grid();
  const WsLayout L = ws_layout(pr, n, H, fp8, grid, group);
  if (!ws || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_CHECK_ARG(aligned16(ws));
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const int esz = fp8 ? 1 : 2;
  const int nt1 = no_mul ? (pr[0].I + 255) / 256 : pr[0].I / 128;  // gemm1 N tiles: 256 gate rows, or 128 gate + 128 up

  // Tiles per unit (host estimate of the unit count from the tile-map bound):
  // one tile per unit, dealt round-robin so tiles sharing a weight tile run side
  // by side -- unless two-tile units of full tiles fill between half a wave and
  // one wave (a deep-K GEMM2): then each weight tile is read once, all units in
  // one wave.  fp8 and several problems use one tile (the fp8 register promotion
  // holds one).  Decode-sized problems (at most 16 slots per expert, K of 32+
  // blocks) may split units across CTAs when there are too few of them for the SMs.
  int mg1 = 1, mg2 = 1;
  bool allow_split = !fp8;
  for (int i = 0; i < n; ++i) allow_split = allow_split && (long long)pr[i].T * pr[i].top_k <= 16LL * pr[i].E;
  if (n == 1 && !fp8) {
    const long long S = (long long)pr[0].T * pr[0].top_k;
    const int cap_tiles = std::max(1, moe_tile_map_capacity((int)S, pr[0].E, BM));
    const bool full_tiles = S >= (long long)BM * pr[0].E;  // experts average a full 128-row tile or more
    // also prefill-sized problems (four or more waves of two-tile units) with deep K loops
    // (64+ blocks): the weight tile goes through shared memory once for two M tiles, and
    // the unit's epilogue, not overlapped with MMAs (the two tiles' accumulators take the
    // whole TMEM), is short against its K loop -- Mixtral-like T=4096 / 8192 experts -5 %
    // / -8 %; with short K loops (Qwen3-like, 12-32 blocks) the unhidden epilogues lose 8 %.
    // And one dense expert (a shared expert) with a wave or more of two-tile units: the
    // DeepSeek-like shared expert at T=4096 / 16384 (-1 % on the layer step, whose routed
    // units fill the shared expert's last wave)
    auto mg_for = [&](int nt, int K) {
      const long long units2 = (long long)((cap_tiles + 1) / 2) * nt;  // estimate with two tiles per unit
      const bool one_wave = 2 * units2 >= grid && units2 <= grid;
      const bool prefill = units2 >= 4LL * grid && K / 64 >= 64;
      const bool dense = pr[0].E == 1 && units2 >= grid;
      return (full_tiles && (one_wave || prefill || dense)) ? 2 : 1;
    };
    mg1 = mg_for(nt1, H);
    mg2 = mg_for((H + 255) / 256, pr[0].I);
  }
  const bool split1 = allow_split && H / 64 >= 32, split2 = allow_split && pr[0].I / 64 >= 32;
  // decode-sized bf16 problems (at most 32 slots each, so no tile holds more than 32 rows):
  // the GEMMs' decode stages (32-row A boxes, six stages)
  bool dec = !fp8;
  for (int i = 0; i < n; ++i) dec = dec && (long long)pr[i].T * pr[i].top_k <= 32;

  GemmMaps maps1[kMaxProblems] = {}, maps2[kMaxProblems] = {};
  GemmProblems g1 = {}, g2 = {};
  g1.nprob = g2.nprob = n;
  int* flags_all = reinterpret_cast<int*>(wsb + L.flags);
  int* ctrs = reinterpret_cast<int*>(wsb + L.ctrs);
  bool ctrs_cleared = false;  // by the plan launch or the first gather launch, else by a memset below
  // The split flags are cleared by the plan launch when there is one (two-tile group
  // maps), else by the first gather launch, else by a plan launch of their own.
  bool gathers = fp8;
  for (int i = 0; i < n; ++i) gathers = gathers || pr[i].sorted_slot != nullptr;
  const bool split = split1 || split2;
  bool flags_pending = split && !(mg1 == 2 || mg2 == 2) && gathers;
  if (mg1 == 2 || mg2 == 2 || (split && !gathers)) {
    // clears every problem's flags; builds problem 0's two-tile group maps (n == 1 when mg > 1)
    const ProbLayout& P = L.p[0];
    plan_kernel<<<1, 1024, 0, s>>>(pr[0].tile_map, pr[0].num_tiles, pr[0].expert_offsets, mg1, mg2,
                                   reinterpret_cast<int32_t*>(wsb + P.gmap), reinterpret_cast<int32_t*>(wsb + P.ngroups),
                                   reinterpret_cast<int32_t*>(wsb + P.gmap2), reinterpret_cast<int32_t*>(wsb + P.ngroups2),
                                   flags_all, L.nflags + 2);  // (the unit counters follow the flags)
    ctrs_cleared = true;
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  for (int i = 0; i < n; ++i) {
    const moe_experts_problem& q = pr[i];
    const ProbLayout& P = L.p[i];
    const long long S = (long long)q.T * q.top_k;
    const int I = q.I, E = q.E;
    const bool gather_rows = q.sorted_slot != nullptr;
    const void* A = gather_rows ? (const void*)(wsb + P.A) : q.a1q;
    float* As = fp8 ? reinterpret_cast<float*>(wsb + P.As) : nullptr;
    void* h = wsb + P.h;
    float* hs = fp8 ? reinterpret_cast<float*>(wsb + P.hs) : nullptr;
    if (gather_rows || fp8) {
      const unsigned gb = (unsigned)((S + 7) / 8);
      gather_kernel<<<gb, 256, 0, s>>>(static_cast<const uint8_t*>(q.a1q), q.a1q_scale, q.sorted_slot, (int)S,
                                       q.top_k, H * esz, hb16 ? 1 : H / 128, gather_rows ? wsb + P.A : nullptr, As,
                                       P.s_pad, group == 128 ? H / 128 : (group == MOE_GROUP_TOKEN ? 1 : 0),
                                       // the split flags when pending, and the unit counters
                                       ctrs_cleared ? nullptr : (flags_pending ? flags_all : ctrs),
                                       ctrs_cleared ? 0 : (flags_pending ? L.nflags : 0) + 2, nullptr, 0, nullptr);
      flags_pending = false;
      ctrs_cleared = true;
      if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    }
    // A maps with one-tile and two-tile boxes; weight maps with 256-row boxes (gemm2:
    // the last N tile of an expert with H % 256 == 128 reads 128 rows past it, which
    // land in discarded output columns, zero-filled past the last expert)
    const bool b1_ok = no_mul ? make_map(&maps1[i].b, q.w13, fp8, H, (long long)E * I, 256)
                              : make_map_gate_up(&maps1[i].b, q.w13, fp8, H, I, E);
    const int a_box = dec ? 32 : 128;
    if (!b1_ok || !make_map(&maps1[i].a, A, fp8, H, S, a_box) || !make_map(&maps1[i].a2, A, fp8, H, S, 256) ||
        !make_map(&maps2[i].a, h, fp8, I, S, a_box) || !make_map(&maps2[i].a2, h, fp8, I, S, 256) ||
        !make_map(&maps2[i].b, q.w2, fp8, I, (long long)E * H, 256))
      return MOE_ERR_CUDA;

    GemmParams& p1 = g1.p[i];
    p1.offsets = q.expert_offsets;
    p1.group_map = mg1 == 2 ? reinterpret_cast<int32_t*>(wsb + P.gmap) : q.tile_map;
    p1.num_groups = mg1 == 2 ? reinterpret_cast<int32_t*>(wsb + P.ngroups) : q.num_tiles;
    p1.sorted_slot = q.sorted_slot;
    p1.K = H;
    p1.NT = nt1;
    p1.I = I;
    p1.H = H;
    p1.b_rows = no_mul ? I : 2 * I;
    p1.s_pad = P.s_pad;
    p1.a_kstride = hb16 ? 0 : P.s_pad;  // "A"/"T": one scale per row for every K block
    p1.a_scale_t = As;
    p1.w_scale = q.w13_scale;
    p1.out = hb16 ? (void*)(wsb + P.hb) : h;
    p1.out_scale_t = hb16 ? nullptr : hs;
    p1.flags = reinterpret_cast<int*>(wsb + P.flags1);
    p1.partials = reinterpret_cast<float*>(wsb + L.partials);
    p1.allow_split = split1;

    GemmParams& p2 = g2.p[i];
    p2 = p1;
    p2.group_map = mg2 == 2 ? reinterpret_cast<int32_t*>(wsb + P.gmap2) : q.tile_map;
    p2.num_groups = mg2 == 2 ? reinterpret_cast<int32_t*>(wsb + P.ngroups2) : q.num_tiles;
    p2.K = I;
    p2.NT = (H + 255) / 256;
    p2.b_rows = H;
    p2.a_scale_t = hs;
    p2.w_scale = q.w2_scale;
    p2.out = q.fused_expert_output;
    p2.out_scale_t = nullptr;
    p2.flags = reinterpret_cast<int*>(wsb + P.flags2);
    p2.allow_split = split2;  // (K of at least 32 blocks for a split to pay)
    // units handed out from a counter (the dynamic schedule of gemm_body) when dealt
    // round-robin
    p1.unit_ctr = i == 0 ? ctrs : nullptr;
    p2.unit_ctr = i == 0 ? ctrs + 1 : nullptr;
  }

  // (no plan and no gather launch: the identity case, e.g. a shared expert alone)
  if (!ctrs_cleared && cudaMemsetAsync(ctrs, 0, 2 * sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t e;
  if (fp8) {  // one problem
    const moe_experts_problem& q = pr[0];
    const ProbLayout& P = L.p[0];
    e = hb16 ? launch_gemm1<true, 1, true>(activation, maps1, g1, grid, s)
             : launch_gemm1<true, 1>(activation, maps1, g1, grid, s);
    if (e == cudaSuccess && hb16) {
      const long long S = (long long)q.T * q.top_k;
      const auto* hbp = reinterpret_cast<const __nv_bfloat16*>(wsb + P.hb);
      uint8_t* hq = wsb + P.h;
      float* hs = reinterpret_cast<float*>(wsb + P.hs);
      if (group == MOE_GROUP_TOKEN) {
        hquant_token_kernel<<<(unsigned)S, 256, 0, s>>>(hbp, q.I, q.expert_offsets, q.E, hq, hs);
      } else {
        unsigned* amax = reinterpret_cast<unsigned*>(wsb + P.hamax);
        e = cudaMemsetAsync(amax, 0, sizeof(unsigned), s);
        const long long nvec = S * (q.I / 8);
        const unsigned gb = (unsigned)((nvec + 255) / 256);
        if (e == cudaSuccess) {
          hquant_tensor_amax_kernel<<<std::min<unsigned>(gb, 4u * grid), 256, 0, s>>>(hbp, q.I, q.expert_offsets, q.E,
                                                                                     amax);
          hquant_tensor_kernel<<<gb, 256, 0, s>>>(hbp, q.I, q.expert_offsets, q.E, amax, hq, hs);
        }
      }
      if (e == cudaSuccess) e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = launch_gemm<true, kGemm2, 1, 0>(maps2, g2, grid, s);
  } else {
    e = dec         ? launch_gemm1<false, 1, false, false, true>(activation, maps1, g1, grid, s)
        : mg1 == 1 ? launch_gemm1<false, 1>(activation, maps1, g1, grid, s)
                   : launch_gemm1<false, 2>(activation, maps1, g1, grid, s);
    if (e == cudaSuccess)
      e = dec         ? launch_gemm<false, kGemm2, 1, 0, false, false, true>(maps2, g2, grid, s)
          : mg2 == 1 ? launch_gemm<false, kGemm2, 1, 0>(maps2, g2, grid, s)
                     : launch_gemm<false, kGemm2, 2, 0>(maps2, g2, grid, s);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_experts_problem one_problem(const void* a1q, const float* a1q_scale, const void* w13, const float* w13_scale,
                                const void* w2, const float* w2_scale, const int32_t* expert_offsets,
                                const int32_t* sorted_slot, const int32_t* tile_map, const int32_t* num_tiles, int T,
                                int I, int E, int top_k, void* out) {
  moe_experts_problem q;
  q.a1q = a1q;
  q.a1q_scale = a1q_scale;
  q.w13 = w13;
  q.w13_scale = w13_scale;
  q.w2 = w2;
  q.w2_scale = w2_scale;
  q.expert_offsets = expert_offsets;
  q.sorted_slot = sorted_slot;
  q.tile_map = tile_map;
  q.num_tiles = num_tiles;
  q.T = T;
  q.I = I;
  q.E = E;
  q.top_k = top_k;
  q.fused_expert_output = out;
  return q;
}

// ------------------------------------------------------------------ single-launch layer
// One cooperative launch runs the whole bf16 layer step for decode-sized problems:
// route -> align -> prepare -> gather -> GEMM1 -> GEMM2 -> finalize, each phase over
// the whole grid (one CTA per SM), separated by grid-wide barriers.  The GEMM phases
// are the persistent GEMM of the separate calls (gemm_body), carrying the routed
// experts and, when the layer has one, the shared expert in the same units.
constexpr int kFusedMaxSlots = 2048;  // T * top_k handled by the one-CTA align
constexpr int kFusedMaxE = 256;       // the router keeps E / 32 <= 8 logits per lane
constexpr int kFusedMaxVec = 8;       // finalize: H / 8 <= 8 vectors per thread
constexpr int kFusedThreads = Warps<false>::THREADS;

struct FusedParams {
  const float* logits;
  const __nv_bfloat16* a1;
  const __nv_bfloat16* residual;    // [T, H] or null
  const __nv_bfloat16* rms_weight;  // [H] or null
  int T, H, I, E, top_k, scoring, weight_on_input, has_shared;
  float eps;
  int32_t* topk_ids;
  float* topk_weights;
  __nv_bfloat16* out;        // [T, H]
  unsigned* grid_ctr;        // barrier arrivals (zeroed before the launch)
  int32_t* offsets;          // routed alignment: [E + 1]
  int32_t* sorted_slot;      // [S]
  int32_t* tile_map;         // [cap][2]
  int32_t* num_tiles;        // [1]
  int32_t* sh_offsets;       // shared expert: [2]
  int32_t* sh_tile_map;      // [ceil(T/128)][2]
  int32_t* sh_num_tiles;     // [1]
  __nv_bfloat16* a1q;        // weight-on-input rows [T, H] (null: the experts read a1)
  __nv_bfloat16* A;          // gathered rows [S, H]
  __nv_bfloat16* y;          // routed expert rows [S, H], token-major
  __nv_bfloat16* ys;         // shared expert rows [T, H]
};

// Grid-wide barrier number `n` (1, 2, ...): every CTA arrives once per barrier on a
// counter zeroed before the launch.  Generic-proxy writes before it are made visible
// to the async proxy (the TMA loads of the next phase) on both sides.  Bounded: gives
// up (recording MOE_ERR_TIMEOUT) after the wait limit or when a failure is recorded.
__device__ bool grid_barrier(unsigned* ctr, unsigned n) {
  asm volatile("fence.proxy.async;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    const unsigned target = n * gridDim.x;
    const uint64_t t0 = global_ns();
    while (true) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= target || status_failed()) break;
      if (global_ns() - t0 > kWaitLimitNs) {
        record_timeout();
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
  asm volatile("fence.proxy.async;" ::: "memory");
  return !status_failed();
}

// The alignment of moe_align for S <= kFusedMaxSlots slots, by one CTA: counts,
// offsets and tile bases (warp 0 scans), a stable scatter in slot order (warp 0, 32
// slots per step, ranks among equal experts from __match_any_sync), then the tile map.
__device__ void fused_align(const int32_t* __restrict__ ids, int S, int E, int32_t* offsets, int32_t* sorted_slot,
                            int32_t* tile_map, int32_t* num_tiles, int* cnt, int* cur, int* tb) {
  const int tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int f = tid; f < S; f += blockDim.x) atomicAdd(&cnt[ids[f]], 1);
  __syncthreads();
  if (tid < 32) {
    const int per = (E + 31) / 32, e0 = lane * per, e1 = min(E, e0 + per);
    int rows = 0, tiles = 0;
    for (int e = e0; e < e1; ++e) {
      rows += cnt[e];
      tiles += (cnt[e] + BM - 1) / BM;
    }
    int xr = rows, xt = tiles;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int yr = __shfl_up_sync(0xffffffffu, xr, off), yt = __shfl_up_sync(0xffffffffu, xt, off);
      if (lane >= off) {
        xr += yr;
        xt += yt;
      }
    }
    int r0 = xr - rows, t0 = xt - tiles;
    for (int e = e0; e < e1; ++e) {
      offsets[e] = r0;
      cur[e] = r0;
      tb[e] = t0;
      r0 += cnt[e];
      t0 += (cnt[e] + BM - 1) / BM;
    }
    if (lane == 31) {
      offsets[E] = xr;
      *num_tiles = xt;
    }
  }
  __syncthreads();
  if (tid < 32) {
    for (int base = 0; base < S; base += 32) {
      const int f = base + lane;
      const int e = f < S ? ids[f] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int pos = f < S ? cur[e] + rank : 0;
      __syncwarp();
      if (f < S) {
        sorted_slot[pos] = f;
        if (rank == 0) cur[e] += __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    const int n = (cnt[e] + BM - 1) / BM;
    for (int i = 0; i < n; ++i) {
      tile_map[2 * (tb[e] + i)] = e;
      tile_map[2 * (tb[e] + i) + 1] = offsets[e] + BM * i;
    }
  }
}

// kDec: the GEMM phases with decode stages (at most 32 slots)
template <bool kDec>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_layer_kernel(const __grid_constant__ CUtensorMap g1a, const __grid_constant__ CUtensorMap g1b,
                       const __grid_constant__ CUtensorMap g1a_s, const __grid_constant__ CUtensorMap g1b_s,
                       const __grid_constant__ CUtensorMap g2a, const __grid_constant__ CUtensorMap g2b,
                       const __grid_constant__ CUtensorMap g2a_s, const __grid_constant__ CUtensorMap g2b_s,
                       const __grid_constant__ GemmProblems pp1, const __grid_constant__ GemmProblems pp2,
                       const __grid_constant__ FusedParams fp) {
  extern __shared__ uint8_t smem_raw[];
  const int T = fp.T, H = fp.H, k = fp.top_k, S = T * k;
  const int lane = threadIdx.x & 31, nwarp = blockDim.x / 32;
  const int gwarp = blockIdx.x * nwarp + (threadIdx.x >> 5), gwarps = gridDim.x * nwarp;
  unsigned bar = 0;

  // route (one warp per token); the shared expert's identity tiles
  for (int t = gwarp; t < T; t += gwarps) route_token<kFusedMaxE / 32>(fp.logits, t, fp.E, k, fp.scoring, fp.topk_ids,
                                                                         fp.topk_weights);
  if (fp.has_shared && blockIdx.x == 0) {
    const int nt = (T + BM - 1) / BM;
    for (int i = threadIdx.x; i < nt; i += blockDim.x) {
      fp.sh_tile_map[2 * i] = 0;
      fp.sh_tile_map[2 * i + 1] = BM * i;
    }
    if (threadIdx.x == 0) {
      fp.sh_offsets[0] = 0;
      fp.sh_offsets[1] = T;
      *fp.sh_num_tiles = nt;
    }
  }
  grid_barrier(fp.grid_ctr, ++bar);

  // align (CTA 0) beside the weight on the input (the other CTAs)
  if (!status_failed()) {
    if (blockIdx.x == 0) {
      int* sm = reinterpret_cast<int*>(smem_raw);
      fused_align(fp.topk_ids, S, fp.E, fp.offsets, fp.sorted_slot, fp.tile_map, fp.num_tiles, sm, sm + kFusedMaxE,
                  sm + 2 * kFusedMaxE);
    }
    if (fp.weight_on_input && (blockIdx.x > 0 || gridDim.x == 1)) {
      const int c0 = gridDim.x == 1 ? 0 : 1, nc = gridDim.x == 1 ? 1 : gridDim.x - 1;
      const long long nvec = (long long)T * H / 8;
      for (long long v = (long long)(blockIdx.x - c0) * blockDim.x + threadIdx.x; v < nvec;
           v += (long long)nc * blockDim.x) {
        const int t = (int)(v * 8 / H);
        // (the weights and every table below were written by earlier phases of this
        // kernel: coherent loads, not the read-only path)
        const float w = __bfloat162float(__float2bfloat16_rn(__ldcg(fp.topk_weights + t)));  // top_k == 1
        float x[8];
        load_bf16x8(fp.a1 + v * 8, x);
        reinterpret_cast<uint4*>(fp.a1q)[v] =
            make_uint4(pack_bf16x2(x[0] * w, x[1] * w), pack_bf16x2(x[2] * w, x[3] * w), pack_bf16x2(x[4] * w, x[5] * w),
                       pack_bf16x2(x[6] * w, x[7] * w));
      }
    }
  }
  grid_barrier(fp.grid_ctr, ++bar);

  // gather: one warp per sorted row
  if (!status_failed()) {
    const __nv_bfloat16* src = fp.weight_on_input ? fp.a1q : fp.a1;
    const int nv = H / 8;
    for (int p = gwarp; p < S; p += gwarps) {
      const int t = __ldcg(fp.sorted_slot + p) / k;
      const uint4* s4 = reinterpret_cast<const uint4*>(src + (size_t)t * H);
      uint4* d4 = reinterpret_cast<uint4*>(fp.A + (size_t)p * H);
      for (int i = lane; i < nv; i += 32) d4[i] = __ldcg(s4 + i);
    }
  }
  grid_barrier(fp.grid_ctr, ++bar);

  // the expert GEMMs (the routed experts and the shared expert in the same units)
  // (after a failed phase the tile maps may be unset: the GEMMs are skipped)
  if (!status_failed())
    gemm_body<false, kGemm1, 1, MOE_ACT_SILU, false, false, true, kDec>(g1a, g1a, g1b, g1a_s, g1a_s, g1b_s, g1a, g1a,
                                                                        pp1, smem_raw, false);
  grid_barrier(fp.grid_ctr, ++bar);
  if (!status_failed())
    gemm_body<false, kGemm2, 1, MOE_ACT_SILU, false, false, true, kDec>(g2a, g2a, g2b, g2a_s, g2a_s, g2b_s, g2a, g2a,
                                                                        pp2, smem_raw, false);
  grid_barrier(fp.grid_ctr, ++bar);

  // finalize: one CTA per token; sums in fp32 (the weighted expert rows, the shared row,
  // the residual), then RMSNorm when a weight is given
  if (status_failed()) return;
  __shared__ float red[kFusedThreads / 32];
  const int nv = H / 8;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    float o[kFusedMaxVec][8];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kFusedMaxVec; ++j) {
      const int v = threadIdx.x + j * blockDim.x;
      if (v >= nv) break;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[j][i] = 0.f;
      for (int kk = 0; kk < k; ++kk) {
        const float w = fp.weight_on_input ? 1.0f : __ldcg(fp.topk_weights + (size_t)t * k + kk);
        float x[8];
        load_bf16x8_cg(fp.y + ((size_t)t * k + kk) * H + v * 8, x);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[j][i] = fmaf(w, x[i], o[j][i]);
      }
      if (fp.has_shared) {
        float x[8];
        load_bf16x8_cg(fp.ys + (size_t)t * H + v * 8, x);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[j][i] += x[i];
      }
      if (fp.residual) {
        float x[8];
        load_bf16x8(fp.residual + (size_t)t * H + v * 8, x);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[j][i] += x[i];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(o[j][i], o[j][i], ss);
    }
    float scale = 1.0f;
    if (fp.rms_weight) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (lane == 0) red[threadIdx.x >> 5] = ss;
      __syncthreads();
      float tot = 0.f;
      for (int w = 0; w < nwarp; ++w) tot += red[w];
      __syncthreads();
      scale = rsqrtf(tot / (float)H + fp.eps);
    }
#pragma unroll
    for (int j = 0; j < kFusedMaxVec; ++j) {
      const int v = threadIdx.x + j * blockDim.x;
      if (v >= nv) break;
      float g[8];
      if (fp.rms_weight) {
        load_bf16x8(fp.rms_weight + v * 8, g);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[j][i] *= scale * g[i];
      }
      reinterpret_cast<uint4*>(fp.out + (size_t)t * H)[v] =
          make_uint4(pack_bf16x2(o[j][0], o[j][1]), pack_bf16x2(o[j][2], o[j][3]), pack_bf16x2(o[j][4], o[j][5]),
                     pack_bf16x2(o[j][6], o[j][7]));
    }
  }
}

// Workspace of the single-launch layer (the counter and the split flags first: one
// memset clears them).
struct FusedLayout {
  size_t ctr, flags1, flags2, ctl_end, offsets, sorted, tiles, ntiles, sh_offsets, sh_tiles, sh_ntiles, a1q, A, h, hs, y,
      ys, partials, total;
  int nflags1, nflags2;
};

FusedLayout fused_layout(int T, int H, int I, int E, int top_k, bool shared, int grid) {
  FusedLayout L{};
  const long long S = (long long)T * top_k;
  const int cap = std::max(1, moe_tile_map_capacity((int)S, E, BM));
  const int sh_tiles = std::max(1, (T + BM - 1) / BM);
  L.nflags1 = (cap + (shared ? sh_tiles : 0)) * (I / 128);
  L.nflags2 = (cap + (shared ? sh_tiles : 0)) * ((H + 255) / 256);
  size_t off = 0;
  L.ctr = off;  // the grid barrier's arrival count, then the two GEMM phases' unit counters
  off += 16;
  L.flags1 = off;
  off += (size_t)L.nflags1 * 4;
  L.flags2 = off;
  off += (size_t)L.nflags2 * 4;
  L.ctl_end = off;
  off = al256(off);
  L.offsets = off;
  off = al256(off + (size_t)(E + 1) * 4);
  L.sorted = off;
  off = al256(off + (size_t)S * 4);
  L.tiles = off;
  off = al256(off + (size_t)cap * 8);
  L.ntiles = off;
  off = al256(off + 4);
  L.sh_offsets = off;
  off = al256(off + 8);
  L.sh_tiles = off;
  off = al256(off + (size_t)sh_tiles * 8);
  L.sh_ntiles = off;
  off = al256(off + 4);
  L.a1q = off;
  off = al256(off + (size_t)T * H * 2);
  L.A = off;
  off = al256(off + (size_t)S * H * 2);
  L.h = off;
  off = al256(off + (size_t)S * I * 2);
  L.hs = off;
  off = al256(off + (shared ? (size_t)T * I * 2 : 0));
  L.y = off;
  off = al256(off + (size_t)S * H * 2);
  L.ys = off;
  off = al256(off + (shared ? (size_t)T * H * 2 : 0));
  L.partials = off;
  off = al256(off + (size_t)grid * BM * BN * 4);
  L.total = off;
  return L;
}

// ------------------------------------------------------------------ batched activation format
// The experts on the batched format ("Fused MoE Kernel Features": the prepare output is
// "standard" or "batched"; "Fused Experts Kernels" lists batched entry points): one slab
// per expert [E, max_tokens, H] with a row count per expert.  The slabs are the GEMMs'
// rows in place (expert e's rows start at e * max_tokens), so there is no gather of rows;
// a plan launch writes the slab bases, the counts clamped to max_tokens and the tile map
// of the counted rows, and the GEMMs are those of moe_experts, ending each expert's rows
// at its count.  The output rows take the same places in an [E, max_tokens, H] output.
__global__ void __launch_bounds__(1024)
    batched_plan_kernel(const int32_t* __restrict__ counts_in, int E, int max_tokens, int32_t* __restrict__ offsets,
                        int32_t* __restrict__ counts, int32_t* __restrict__ tile_map, int32_t* __restrict__ num_tiles,
                        int* __restrict__ flags, int nflags) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < nflags; i += 1024) flags[i] = 0;
  if (threadIdx.x == 0) carry = 0;
  for (int e = threadIdx.x; e <= E; e += 1024) offsets[e] = e * max_tokens;
  __syncthreads();
  for (int base = 0; base < E; base += 1024) {
    const int e = base + threadIdx.x;
    int c = 0;
    if (e < E) {
      c = min(max(counts_in[e], 0), max_tokens);
      counts[e] = c;
    }
    const int nt = (c + BM - 1) / BM;
    int x = nt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const int w = warp_tot[lane];
      int wx = w;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wx, off);
        if (lane >= off) wx += y;
      }
      warp_tot[lane] = wx - w;
    }
    __syncthreads();
    const int first = carry + warp_tot[warp] + x - nt;
    for (int i = 0; i < nt; ++i) {
      tile_map[2 * (first + i)] = e;
      tile_map[2 * (first + i) + 1] = e * max_tokens + i * BM;
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry = first + nt;
    __syncthreads();
  }
  if (threadIdx.x == 0) *num_tiles = carry;
}

struct BatchedLayout {
  WsLayout L;
  size_t offsets, counts, tiles, ntiles, total;
  int cap;
};

BatchedLayout batched_layout(int E, int M, int H, int I, const moe_quant_config* qc, int grid) {
  BatchedLayout B{};
  const moe_experts_problem q = one_problem(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                            nullptr, nullptr, E * M, I, E, 1, nullptr);
  B.L = ws_layout(&q, 1, H, qc->act == MOE_DT_FP8_E4M3, grid, qc->act_group, true);
  B.cap = std::max(1, E * ((M + BM - 1) / BM));
  size_t off = B.L.total;
  B.offsets = off;
  off = al256(off + (size_t)(E + 1) * 4);
  B.counts = off;
  off = al256(off + (size_t)E * 4);
  B.tiles = off;
  off = al256(off + (size_t)B.cap * 8);
  B.ntiles = off;
  off = al256(off + 4);
  B.total = off;
  return B;
}

moe_status_t experts_batched_run(const void* a1q_b, const float* a1q_b_scale, const void* w13, const float* w13_scale,
                                 const void* w2, const float* w2_scale, const int32_t* expert_num_tokens, int E, int M,
                                 int H, int I, const moe_quant_config* qc, int activation, void* out_b, void* ws,
                                 size_t ws_bytes, cudaStream_t s) {
  MOE_CHECK_ARG(qc && E >= 1 && M >= 1 && H > 0 && I > 0 && H % 128 == 0 && I % 128 == 0);
  if (activation < MOE_ACT_SILU || activation > MOE_ACT_GELU_NO_MUL || !quant_ok(qc)) return MOE_ERR_UNSUPPORTED;
  MOE_CHECK_ARG(fits_int32((long long)E * M + 4 * BM) && fits_int32((long long)E * 2 * I) &&
                fits_int32((long long)E * H) && fits_int32((long long)H * 8));
  const bool fp8 = qc->act == MOE_DT_FP8_E4M3;
  const int group = qc->act_group;
  const bool hb16 = fp8 && group != 128;
  const bool no_mul = activation == MOE_ACT_SILU_NO_MUL || activation == MOE_ACT_GELU_NO_MUL;
  MOE_CHECK_ARG(a1q_b && w13 && w2 && expert_num_tokens && out_b);
  MOE_CHECK_ARG(!fp8 || (a1q_b_scale && w13_scale && w2_scale));
  MOE_CHECK_ARG(aligned16(a1q_b) && aligned16(w13) && aligned16(w2) && aligned16(out_b));
  const int grid = gemm_grid();
  const BatchedLayout B = batched_layout(E, M, H, I, qc, grid);
  if (!ws || ws_bytes < B.total) return MOE_ERR_WORKSPACE;
  MOE_CHECK_ARG(aligned16(ws));
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const ProbLayout& P = B.L.p[0];
  const long long S = (long long)E * M;
  auto* offsets = reinterpret_cast<int32_t*>(wsb + B.offsets);
  auto* counts = reinterpret_cast<int32_t*>(wsb + B.counts);
  auto* tiles = reinterpret_cast<int32_t*>(wsb + B.tiles);
  auto* ntiles = reinterpret_cast<int32_t*>(wsb + B.ntiles);
  batched_plan_kernel<<<1, 1024, 0, s>>>(expert_num_tokens, E, M, offsets, counts, tiles, ntiles,
                                         reinterpret_cast<int*>(wsb + B.L.flags), B.L.nflags);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  float* As = fp8 ? reinterpret_cast<float*>(wsb + P.As) : nullptr;
  if (fp8) {
    // the slabs' activation scales transposed to [K/128][rows] (no rows move)
    gather_kernel<<<(unsigned)((S + 7) / 8), 256, 0, s>>>(
        nullptr, a1q_b_scale, nullptr, (int)S, 1, 0, hb16 ? 1 : H / 128, nullptr, As, P.s_pad,
        group == 128 ? H / 128 : (group == MOE_GROUP_TOKEN ? 1 : 0), nullptr, 0, nullptr, 0, nullptr);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  void* h = wsb + P.h;
  float* hs = fp8 ? reinterpret_cast<float*>(wsb + P.hs) : nullptr;
  GemmMaps m1 = {}, m2 = {};
  const int a2_rows = 256;
  const bool b1_ok = no_mul ? make_map(&m1.b, w13, fp8, H, (long long)E * I, 256) : make_map_gate_up(&m1.b, w13, fp8, H, I, E);
  if (!b1_ok || !make_map(&m1.a, a1q_b, fp8, H, S, 128) || !make_map(&m1.a2, a1q_b, fp8, H, S, a2_rows) ||
      !make_map(&m2.a, h, fp8, I, S, 128) || !make_map(&m2.a2, h, fp8, I, S, a2_rows) ||
      !make_map(&m2.b, w2, fp8, I, (long long)E * H, 256))
    return MOE_ERR_CUDA;
  GemmProblems g1 = {}, g2 = {};
  g1.nprob = g2.nprob = 1;
  GemmParams& p1 = g1.p[0];
  p1.offsets = offsets;
  p1.counts = counts;
  p1.group_map = tiles;
  p1.num_groups = ntiles;
  p1.sorted_slot = nullptr;
  p1.K = H;
  p1.NT = no_mul ? (I + 255) / 256 : I / 128;
  p1.I = I;
  p1.H = H;
  p1.b_rows = no_mul ? I : 2 * I;
  p1.s_pad = P.s_pad;
  p1.a_kstride = hb16 ? 0 : P.s_pad;
  p1.a_scale_t = As;
  p1.w_scale = w13_scale;
  p1.out = hb16 ? (void*)(wsb + P.hb) : h;
  p1.out_scale_t = hb16 ? nullptr : hs;
  p1.flags = reinterpret_cast<int*>(wsb + P.flags1);
  p1.partials = reinterpret_cast<float*>(wsb + B.L.partials);
  p1.allow_split = 0;
  GemmParams& p2 = g2.p[0];
  p2 = p1;
  p2.K = I;
  p2.NT = (H + 255) / 256;
  p2.b_rows = H;
  p2.a_scale_t = hs;
  p2.w_scale = w2_scale;
  p2.out = out_b;
  p2.out_scale_t = nullptr;
  p2.flags = reinterpret_cast<int*>(wsb + P.flags2);
  cudaError_t e;
  if (fp8) {
    if (hb16 && group == MOE_GROUP_TENSOR &&
        cudaMemsetAsync(wsb + P.hb, 0, (size_t)S * I * 2, s) != cudaSuccess)  // uncounted rows: no amax
      return MOE_ERR_CUDA;
    e = hb16 ? launch_gemm1<true, 1, true>(activation, &m1, g1, grid, s) : launch_gemm1<true, 1>(activation, &m1, g1, grid, s);
    if (e == cudaSuccess && hb16) {
      const auto* hbp = reinterpret_cast<const __nv_bfloat16*>(wsb + P.hb);
      uint8_t* hq = wsb + P.h;
      if (group == MOE_GROUP_TOKEN) {
        hquant_token_kernel<<<(unsigned)S, 256, 0, s>>>(hbp, I, offsets, E, hq, hs);
      } else {
        unsigned* amax = reinterpret_cast<unsigned*>(wsb + P.hamax);
        e = cudaMemsetAsync(amax, 0, sizeof(unsigned), s);
        const long long nvec = S * (I / 8);
        const unsigned gb = (unsigned)((nvec + 255) / 256);
        if (e == cudaSuccess) {
          hquant_tensor_amax_kernel<<<std::min<unsigned>(gb, 4u * grid), 256, 0, s>>>(hbp, I, offsets, E, amax);
          hquant_tensor_kernel<<<gb, 256, 0, s>>>(hbp, I, offsets, E, amax, hq, hs);
        }
      }
      if (e == cudaSuccess) e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = launch_gemm<true, kGemm2, 1, 0>(&m2, g2, grid, s);
  } else {
    e = launch_gemm1<false, 1>(activation, &m1, g1, grid, s);
    if (e == cudaSuccess) e = launch_gemm<false, kGemm2, 1, 0>(&m2, g2, grid, s);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ------------------------------------------------------------------ NVFP4 experts
// Workspace of an NVFP4 call: gathered A rows and their scale rows, the bf16
// intermediate, its NVFP4 codes and scales, the split flags of both GEMMs and one
// split partial per CTA.
struct Fp4Layout {
  size_t A, ASF, hb, hq, hsf, flags, partials, total;
  int nflags1, nflags2;
};

Fp4Layout ws_layout_nvfp4(long long S, int H, int I, int E, int grid) {
  Fp4Layout L{};
  const int cap_groups = std::max(1, moe_tile_map_capacity((int)S, E, BM));
  L.nflags1 = cap_groups * (I / 128);
  L.nflags2 = cap_groups * (H / 256);
  size_t off = 0;
  L.A = off;
  off = al256(off + (size_t)S * H / 2);
  L.ASF = off;
  off = al256(off + (size_t)S * H / 16);
  L.hb = off;
  off = al256(off + (size_t)S * I * 2);
  L.hq = off;
  off = al256(off + (size_t)S * I / 2);
  L.hsf = off;
  off = al256(off + (size_t)S * I / 16);
  L.flags = off;
  off = al256(off + (size_t)(L.nflags1 + L.nflags2) * 4);
  L.partials = off;
  off = al256(off + (size_t)grid * BM * BN * 4);
  L.total = off;
  return L;
}

// gather (+ scale rows) -> gemm1 (bf16 h) -> NVFP4 quantisation of h -> gemm2
moe_status_t experts_nvfp4_run(const void* a1q, const void* a1q_sf, const float* a1_gscale, const void* w13,
                               const void* w13_sf, const float* w13_gscale, const void* w2, const void* w2_sf,
                               const float* w2_gscale, const float* h_gscale, const int32_t* expert_offsets,
                               const int32_t* sorted_slot, const int32_t* tile_map, const int32_t* num_tiles, int T,
                               int H, int I, int E, int top_k, int activation, void* out, void* ws, size_t ws_bytes,
                               cudaStream_t s) {
  if (activation < MOE_ACT_SILU || activation > MOE_ACT_GELU_NO_MUL) return MOE_ERR_UNSUPPORTED;
  MOE_CHECK_ARG(T >= 0 && H > 0 && H % 256 == 0 && I > 0 && I % 256 == 0 && E >= 1 && top_k >= 1 && top_k <= E);
  const long long S = (long long)T * top_k;
  MOE_CHECK_ARG(fits_int32(S + 4 * BM) && fits_int32((long long)E * 2 * I) && fits_int32((long long)E * H) &&
                fits_int32((long long)H * 8));
  if (S == 0) return MOE_OK;
  MOE_CHECK_ARG(a1q && a1q_sf && a1_gscale && w13 && w13_sf && w13_gscale && w2 && w2_sf && w2_gscale && h_gscale &&
                expert_offsets && tile_map && num_tiles && out);
  MOE_CHECK_ARG(sorted_slot || (E == 1 && top_k == 1));
  MOE_CHECK_ARG(aligned16(a1q) && aligned16(a1q_sf) && aligned16(w13) && aligned16(w13_sf) && aligned16(w2) &&
                aligned16(w2_sf) && aligned16(out));
  const bool no_mul = activation == MOE_ACT_SILU_NO_MUL || activation == MOE_ACT_GELU_NO_MUL;
  const int grid = gemm_grid();
  const Fp4Layout L = ws_layout_nvfp4(S, H, I, E, grid);
  if (!ws || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_CHECK_ARG(aligned16(ws));
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  // decode-sized problems split units across CTAs, as in the bf16 path
  const bool allow_split = S <= 16LL * E;
  const bool split1 = allow_split && H / 64 >= 32, split2 = allow_split && I / 64 >= 32;
  int* flags = reinterpret_cast<int*>(wsb + L.flags);
  const int nflags = L.nflags1 + L.nflags2;
  const bool split = split1 || split2;
  const bool gather_rows = sorted_slot != nullptr;
  if (gather_rows) {
    gather_kernel<<<(unsigned)((S + 7) / 8), 256, 0, s>>>(
        static_cast<const uint8_t*>(a1q), nullptr, sorted_slot, (int)S, top_k, H / 2, 0, wsb + L.A, nullptr, 0, 0,
        split ? flags : nullptr, split ? nflags : 0, static_cast<const uint8_t*>(a1q_sf), H / 16, wsb + L.ASF);
  } else if (split) {
    plan_kernel<<<1, 1024, 0, s>>>(tile_map, num_tiles, expert_offsets, 1, 1, nullptr, nullptr, nullptr, nullptr,
                                   flags, nflags);
  }
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  const void* A = gather_rows ? (const void*)(wsb + L.A) : a1q;
  const void* ASF = gather_rows ? (const void*)(wsb + L.ASF) : a1q_sf;
  void* hb = wsb + L.hb;
  uint8_t* hq = wsb + L.hq;
  uint8_t* hsf = wsb + L.hsf;
  // packed operands are uint8 maps over rows of K/2 bytes; scale rows are K/16 bytes
  // (at most 32 slots: the decode stages, 32-row A and A-scale boxes)
  const bool dec = S <= 32;
  const int a_box = dec ? 32 : 128;
  GemmMaps m1 = {}, m2 = {};
  const bool b1 = no_mul ? make_map(&m1.b, w13, true, H / 2, (long long)E * I, 256)
                         : make_map_gate_up(&m1.b, w13, true, H / 2, I, E);
  const bool sb1 = no_mul ? make_map_sf(&m1.sb, w13_sf, H / 16, (long long)E * I, 256)
                          : make_map_sf_gate_up(&m1.sb, w13_sf, H / 16, I, E);
  if (!b1 || !sb1 || !make_map(&m1.a, A, true, H / 2, S, a_box) || !make_map(&m1.a2, A, true, H / 2, S, 128) ||
      !make_map_sf(&m1.sa, ASF, H / 16, S, a_box) || !make_map(&m2.a, hq, true, I / 2, S, a_box) ||
      !make_map(&m2.a2, hq, true, I / 2, S, 128) || !make_map_sf(&m2.sa, hsf, I / 16, S, a_box) ||
      !make_map(&m2.b, w2, true, I / 2, (long long)E * H, 256) ||
      !make_map_sf(&m2.sb, w2_sf, I / 16, (long long)E * H, 256))
    return MOE_ERR_CUDA;

  GemmProblems g1 = {}, g2 = {};
  g1.nprob = g2.nprob = 1;
  GemmParams& p1 = g1.p[0];
  p1.offsets = expert_offsets;
  p1.group_map = tile_map;
  p1.num_groups = num_tiles;
  p1.sorted_slot = sorted_slot;
  p1.K = H;
  p1.NT = no_mul ? (I + 255) / 256 : I / 128;
  p1.I = I;
  p1.H = H;
  p1.b_rows = no_mul ? I : 2 * I;
  p1.a_gscale = a1_gscale;
  p1.w_gscale = w13_gscale;
  p1.out = hb;
  p1.flags = flags;
  p1.partials = reinterpret_cast<float*>(wsb + L.partials);
  p1.allow_split = split1;
  GemmParams& p2 = g2.p[0];
  p2 = p1;
  p2.K = I;
  p2.NT = H / 256;
  p2.b_rows = H;
  p2.a_gscale = h_gscale;
  p2.w_gscale = w2_gscale;
  p2.out = out;
  p2.flags = flags + L.nflags1;
  p2.allow_split = split2;

  cudaError_t e = dec ? launch_gemm1<false, 1, false, true, true>(activation, &m1, g1, grid, s)
                      : launch_gemm1<false, 1, false, true>(activation, &m1, g1, grid, s);
  if (e == cudaSuccess) {
    const long long groups = S * (I / 16);
    nvfp4_quant_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(hb), I, S,
                                                                        expert_offsets + E, nullptr, h_gscale, hq,
                                                                        hsf);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess)
    e = dec ? launch_gemm<false, kGemm2, 1, 0, false, true, true>(&m2, g2, grid, s)
            : launch_gemm<false, kGemm2, 1, 0, false, true>(&m2, g2, grid, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Self-test of the failure path of the device-side waits: one thread waits (bounded) on an
// mbarrier that no thread arrives on, with the GEMMs' wait routine and a caller-chosen
// limit; the wait gives up, records MOE_ERR_TIMEOUT and the kernel returns.
// div_rn_by against __fdiv_rn on n (dividend, divisor) pairs drawn from a counter-based
// hash: divisors are the requantisation scales max(amax, 1e-10) / 448 of amax values over
// 2^-40 .. 2^40 (with every mantissa), dividends of either sign anywhere in [0, amax]
// (their mantissas and exponents drawn independently, zeros included), and every
// mismatching bit pattern is counted into *mismatches (which the caller zeroes).
__device__ __forceinline__ uint32_t selftest_hash(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352dU;
  x ^= x >> 15;
  x *= 0x846ca68bU;
  x ^= x >> 16;
  return x;
}
__global__ void __launch_bounds__(256)
    division_selftest_kernel(long long n, uint32_t seed, unsigned long long* mismatches) {
  unsigned long long bad = 0;
  for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n; i += (long long)gridDim.x * 256) {
    const uint32_t h0 = selftest_hash((uint32_t)i * 2u + 1u + seed * 0x9e3779b9U);
    const uint32_t h1 = selftest_hash(h0 ^ 0x5bd1e995U);
    const uint32_t h2 = selftest_hash(h1 + (uint32_t)(i >> 32));
    // amax = mantissa (23 random bits) x 2^(e - 40), e in [0, 80]
    const float amax = __uint_as_float(((h0 % 81u + 87u) << 23) | (h1 & 0x7FFFFFu));
    const float s = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
    // x = +-(random mantissa) x 2^-k x amax-scale, k in [0, 40); 1 in 64 exactly 0 or amax
    float x = __uint_as_float(((h2 % 40u + 87u) << 23) | (h2 >> 9 & 0x7FFFFFu));
    x = fminf(__fmul_rn(x, __uint_as_float(__float_as_uint(amax) & 0x7F800000u)), amax);  // x amax's power of 2
    if ((h1 >> 23 & 63u) == 0u) x = (h1 & (1u << 30)) ? amax : 0.0f;
    if (h2 & 1u) x = -x;
    const float q_ref = __fdiv_rn(x, s);
    const float q = div_rn_by(x, s, __frcp_rn(s));
    if (__float_as_uint(q) != __float_as_uint(q_ref)) ++bad;
  }
  if (bad) atomicAdd(mismatches, bad);
}

__global__ void __launch_bounds__(32) selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    mbar_wait(&bar, 0, false, limit_ns);  // phase 0 never completes: no arrival
    mbar_inval(&bar);
  }
}

}  // namespace

MOE_DEFINE_STATUS_READER(experts_status)

}  // namespace moe

using namespace moe;

extern "C" size_t moe_workspace_size(int T, int H, int I, int E, int top_k, const moe_quant_config* qc) {
  if (!qc || T < 0 || H <= 0 || I <= 0 || E < 1 || top_k < 1) return 0;
  const moe_experts_problem q = one_problem(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                            nullptr, nullptr, T, I, E, top_k, nullptr);
  return ws_layout(&q, 1, H, qc->act == MOE_DT_FP8_E4M3, gemm_grid(), qc->act_group).total;
}

extern "C" moe_status_t moe_workspace_intermediate(int T, int H, int I, int E, int top_k, const moe_quant_config* qc,
                                                   size_t* h_offset, size_t* h_scale_offset, int* scale_stride) {
  MOE_CHECK_ARG(qc && h_offset && h_scale_offset && scale_stride && T >= 0 && H > 0 && I > 0 && E >= 1 && top_k >= 1);
  if (!quant_ok(qc)) return MOE_ERR_UNSUPPORTED;
  const moe_experts_problem q = one_problem(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                            nullptr, nullptr, T, I, E, top_k, nullptr);
  const bool fp8 = qc->act == MOE_DT_FP8_E4M3;
  const WsLayout L = ws_layout(&q, 1, H, fp8, gemm_grid(), qc->act_group);
  *h_offset = L.p[0].h;
  *h_scale_offset = fp8 ? L.p[0].hs : 0;
  *scale_stride = !fp8 ? 0 : (qc->act_group == 128 ? L.p[0].s_pad : 1);
  return MOE_OK;
}

extern "C" moe_status_t moe_workspace_intermediate_nvfp4(int T, int H, int I, int E, int top_k, size_t* hb_offset,
                                                         size_t* hq_offset, size_t* hsf_offset) {
  MOE_CHECK_ARG(hb_offset && hq_offset && hsf_offset && T >= 0 && H > 0 && H % 256 == 0 && I > 0 && I % 256 == 0 &&
                E >= 1 && top_k >= 1);
  const Fp4Layout L = ws_layout_nvfp4((long long)T * top_k, H, I, E, gemm_grid());
  *hb_offset = L.hb;
  *hq_offset = L.hq;
  *hsf_offset = L.hsf;
  return MOE_OK;
}

extern "C" size_t moe_workspace_size_multi(const moe_experts_problem* problems, int num_problems, int H,
                                           const moe_quant_config* qc) {
  if (!qc || !problems || num_problems < 1 || num_problems > kMaxProblems || H <= 0) return 0;
  for (int i = 0; i < num_problems; ++i)
    if (problems[i].T < 0 || problems[i].I <= 0 || problems[i].E < 1 || problems[i].top_k < 1) return 0;
  return ws_layout(problems, num_problems, H, qc->act == MOE_DT_FP8_E4M3, gemm_grid(), qc->act_group).total;
}

extern "C" moe_status_t moe_experts_multi(const moe_experts_problem* problems, int num_problems, int H,
                                          const moe_quant_config* qc, int activation, void* ws, size_t ws_bytes,
                                          moe_stream_t stream) {
  return experts_run(problems, num_problems, H, qc, activation, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" moe_status_t moe_experts_act(const void* a1q, const float* a1q_scale, const void* w13,
                                        const float* w13_scale, const void* w2, const float* w2_scale,
                                        const int32_t* expert_offsets, const int32_t* sorted_slot,
                                        const int32_t* tile_map, const int32_t* num_tiles, int T, int H, int I, int E,
                                        int top_k, const moe_quant_config* qc, int activation,
                                        void* fused_expert_output, void* ws, size_t ws_bytes, moe_stream_t stream) {
  const moe_experts_problem q = one_problem(a1q, a1q_scale, w13, w13_scale, w2, w2_scale, expert_offsets, sorted_slot,
                                            tile_map, num_tiles, T, I, E, top_k, fused_expert_output);
  return experts_run(&q, 1, H, qc, activation, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" moe_status_t moe_experts(const void* a1q, const float* a1q_scale, const void* w13, const float* w13_scale,
                                    const void* w2, const float* w2_scale, const int32_t* expert_offsets,
                                    const int32_t* sorted_slot, const int32_t* tile_map, const int32_t* num_tiles,
                                    int T, int H, int I, int E, int top_k, const moe_quant_config* qc,
                                    void* fused_expert_output, void* ws, size_t ws_bytes, moe_stream_t stream) {
  return moe_experts_act(a1q, a1q_scale, w13, w13_scale, w2, w2_scale, expert_offsets, sorted_slot, tile_map,
                         num_tiles, T, H, I, E, top_k, qc, MOE_ACT_SILU, fused_expert_output, ws, ws_bytes, stream);
}

extern "C" size_t moe_workspace_size_nvfp4(int T, int H, int I, int E, int top_k) {
  if (T < 0 || H <= 0 || H % 256 || I <= 0 || I % 256 || E < 1 || top_k < 1) return 0;
  return ws_layout_nvfp4((long long)T * top_k, H, I, E, gemm_grid()).total;
}

extern "C" moe_status_t moe_experts_nvfp4(const void* a1q, const void* a1q_sf, const float* a1_gscale,
                                          const void* w13, const void* w13_sf, const float* w13_gscale,
                                          const void* w2, const void* w2_sf, const float* w2_gscale,
                                          const float* h_gscale, const int32_t* expert_offsets,
                                          const int32_t* sorted_slot, const int32_t* tile_map,
                                          const int32_t* num_tiles, int T, int H, int I, int E, int top_k,
                                          int activation, void* fused_expert_output, void* ws, size_t ws_bytes,
                                          moe_stream_t stream) {
  return experts_nvfp4_run(a1q, a1q_sf, a1_gscale, w13, w13_sf, w13_gscale, w2, w2_sf, w2_gscale, h_gscale,
                           expert_offsets, sorted_slot, tile_map, num_tiles, T, H, I, E, top_k, activation,
                           fused_expert_output, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" moe_status_t moe_prepare_nvfp4(const void* a1, const float* topk_weights, int T, int H, int top_k,
                                          int apply_router_weight_on_input, const float* a1_gscale, void* a1q,
                                          void* a1q_sf, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && H > 0 && H % 16 == 0 && top_k >= 1);
  MOE_CHECK_ARG(!apply_router_weight_on_input || (top_k == 1 && topk_weights));
  MOE_CHECK_ARG(fits_int32((long long)H * 8));
  if (T == 0) return MOE_OK;
  MOE_CHECK_ARG(a1 && a1_gscale && a1q && a1q_sf && aligned16(a1) && aligned16(a1q));
  const long long groups = (long long)T * (H / 16);
  nvfp4_quant_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(a1), H, T, nullptr, apply_router_weight_on_input ? topk_weights : nullptr,
      a1_gscale, static_cast<uint8_t*>(a1q), static_cast<uint8_t*>(a1q_sf));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" size_t moe_layer_fused_workspace_size(int T, int H, int I, int E, int top_k, int has_shared) {
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || top_k < 1) return 0;
  return fused_layout(T, H, I, E, top_k, has_shared != 0, gemm_grid()).total;
}

extern "C" moe_status_t moe_layer_fused(const float* logits, const void* a1, int T, int H, int I, int E, int top_k,
                                        int scoring, int apply_router_weight_on_input, const void* w13, const void* w2,
                                        const void* shared_w13, const void* shared_w2, const void* residual,
                                        const void* rms_weight, float eps, int32_t* topk_ids, float* topk_weights,
                                        void* output, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && E >= 1 && top_k >= 1 && top_k <= E && top_k <= 32 && H > 0 && I > 0);
  MOE_CHECK_ARG(scoring == MOE_SCORING_SOFTMAX_RENORM || scoring == MOE_SCORING_SIGMOID);
  MOE_CHECK_ARG(scoring != MOE_SCORING_SIGMOID || top_k == 1);
  MOE_CHECK_ARG(!apply_router_weight_on_input || top_k == 1);
  MOE_CHECK_ARG(H % 128 == 0 && I % 128 == 0 && fits_int32((long long)H * 8) && fits_int32((long long)E * 2 * I));
  MOE_CHECK_ARG((shared_w13 == nullptr) == (shared_w2 == nullptr));
  if ((long long)T * top_k > kFusedMaxSlots || E > kFusedMaxE || H / 8 > kFusedMaxVec * kFusedThreads)
    return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  MOE_CHECK_ARG(logits && a1 && w13 && w2 && topk_ids && topk_weights && output);
  MOE_CHECK_ARG(aligned16(a1) && aligned16(w13) && aligned16(w2) && aligned16(output) &&
                (!shared_w13 || (aligned16(shared_w13) && aligned16(shared_w2))) && (!residual || aligned16(residual)) &&
                (!rms_weight || aligned16(rms_weight)));
  const bool shared = shared_w13 != nullptr;
  const int grid = gemm_grid();
  const FusedLayout L = fused_layout(T, H, I, E, top_k, shared, grid);
  if (!ws || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_CHECK_ARG(aligned16(ws));
  int dev = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!coop) return MOE_ERR_UNSUPPORTED;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const long long S = (long long)T * top_k;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  FusedParams fp{};
  fp.logits = logits;
  fp.a1 = static_cast<const __nv_bfloat16*>(a1);
  fp.residual = static_cast<const __nv_bfloat16*>(residual);
  fp.rms_weight = static_cast<const __nv_bfloat16*>(rms_weight);
  fp.T = T;
  fp.H = H;
  fp.I = I;
  fp.E = E;
  fp.top_k = top_k;
  fp.scoring = scoring;
  fp.weight_on_input = apply_router_weight_on_input != 0;
  fp.has_shared = shared;
  fp.eps = eps;
  fp.topk_ids = topk_ids;
  fp.topk_weights = topk_weights;
  fp.out = static_cast<__nv_bfloat16*>(output);
  fp.grid_ctr = reinterpret_cast<unsigned*>(wsb + L.ctr);
  fp.offsets = reinterpret_cast<int32_t*>(wsb + L.offsets);
  fp.sorted_slot = reinterpret_cast<int32_t*>(wsb + L.sorted);
  fp.tile_map = reinterpret_cast<int32_t*>(wsb + L.tiles);
  fp.num_tiles = reinterpret_cast<int32_t*>(wsb + L.ntiles);
  fp.sh_offsets = reinterpret_cast<int32_t*>(wsb + L.sh_offsets);
  fp.sh_tile_map = reinterpret_cast<int32_t*>(wsb + L.sh_tiles);
  fp.sh_num_tiles = reinterpret_cast<int32_t*>(wsb + L.sh_ntiles);
  fp.a1q = reinterpret_cast<__nv_bfloat16*>(wsb + L.a1q);
  fp.A = reinterpret_cast<__nv_bfloat16*>(wsb + L.A);
  fp.y = reinterpret_cast<__nv_bfloat16*>(wsb + L.y);
  fp.ys = shared ? reinterpret_cast<__nv_bfloat16*>(wsb + L.ys) : nullptr;
  void* h = wsb + L.h;
  void* hs = wsb + L.hs;

  // tensor maps: gemm1 reads the gathered rows and w13 (the shared expert: a1 and its
  // w13), gemm2 the intermediates and w2
  // (at most 32 slots: the decode stages, 32-row A boxes)
  const bool dec = S <= 32;
  const int a_box = dec ? 32 : 128;
  GemmMaps m1[2] = {}, m2[2] = {};
  if (!make_map(&m1[0].a, fp.A, false, H, S, a_box) || !make_map_gate_up(&m1[0].b, w13, false, H, I, E) ||
      !make_map(&m2[0].a, h, false, I, S, a_box) || !make_map(&m2[0].b, w2, false, I, (long long)E * H, 256))
    return MOE_ERR_CUDA;
  if (shared &&
      (!make_map(&m1[1].a, a1, false, H, T, a_box) || !make_map_gate_up(&m1[1].b, shared_w13, false, H, I, 1) ||
       !make_map(&m2[1].a, hs, false, I, T, a_box) || !make_map(&m2[1].b, shared_w2, false, I, H, 256)))
    return MOE_ERR_CUDA;
  if (!shared) {
    m1[1] = m1[0];
    m2[1] = m2[0];
  }
  // the split rule of the separate calls: decode-sized problems with deep K
  const bool allow_split = S <= 16LL * E && (!shared || T <= 16);
  const bool split1 = allow_split && H / 64 >= 32, split2 = allow_split && I / 64 >= 32;
  const int cap = std::max(1, moe_tile_map_capacity((int)S, E, BM));
  GemmProblems g1 = {}, g2 = {};
  g1.nprob = g2.nprob = shared ? 2 : 1;
  for (int i = 0; i < g1.nprob; ++i) {
    GemmParams& q1 = g1.p[i];
    q1.offsets = i ? fp.sh_offsets : fp.offsets;
    q1.group_map = i ? fp.sh_tile_map : fp.tile_map;
    q1.num_groups = i ? fp.sh_num_tiles : fp.num_tiles;
    q1.sorted_slot = i ? nullptr : fp.sorted_slot;
    q1.K = H;
    q1.NT = I / 128;
    q1.I = I;
    q1.H = H;
    q1.b_rows = 2 * I;
    q1.out = i ? hs : h;
    q1.flags = reinterpret_cast<int*>(wsb + L.flags1) + (i ? cap * (I / 128) : 0);
    q1.partials = reinterpret_cast<float*>(wsb + L.partials);
    q1.allow_split = split1;
    GemmParams& q2 = g2.p[i];
    q2 = q1;
    q2.K = I;
    q2.NT = (H + 255) / 256;
    q2.b_rows = H;
    q2.out = i ? (void*)fp.ys : (void*)fp.y;
    q2.flags = reinterpret_cast<int*>(wsb + L.flags2) + (i ? cap * ((H + 255) / 256) : 0);
    q2.allow_split = split2;
    // the GEMM phases' unit counters (dynamic schedule when units go round-robin): the two
    // words after the barrier counter, cleared with it before the launch
    q1.unit_ctr = i == 0 ? reinterpret_cast<int*>(wsb + L.ctr) + 1 : nullptr;
    q2.unit_ctr = i == 0 ? reinterpret_cast<int*>(wsb + L.ctr) + 2 : nullptr;
  }
  static int configured[2][64] = {{0}};
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
               CUtensorMap, GemmProblems, GemmProblems, FusedParams) =
      dec ? fused_layer_kernel<true> : fused_layer_kernel<false>;
  const int smem = dec ? Cfg<false, 1, false, true>::SMEM_BYTES : Cfg<false, 1>::SMEM_BYTES;
  if (dev < 64 && !configured[dec][dev]) {
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(kern), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    configured[dec][dev] = 1;
  }
  // the barrier counter and the split flags start at zero
  if (cudaMemsetAsync(wsb + L.ctr, 0, L.ctl_end - L.ctr, s) != cudaSuccess) return MOE_ERR_CUDA;
  // a cooperative launch: every CTA resident at once (the grid barriers need it), or an error
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(kFusedThreads);
  lc.dynamicSmemBytes = (size_t)smem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, kern, m1[0].a, m1[0].b, m1[1].a, m1[1].b, m2[0].a, m2[0].b, m2[1].a, m2[1].b, g1, g2,
                         fp) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" moe_status_t moe_selftest_row_division(long long n, uint32_t seed, unsigned long long* mismatches,
                                                  moe_stream_t stream) {
  MOE_CHECK_ARG(n >= 0 && mismatches);
  if (n == 0) return MOE_OK;
  division_selftest_kernel<<<(unsigned)std::min<long long>((n + 255) / 256, 4096), 256, 0,
                             reinterpret_cast<cudaStream_t>(stream)>>>(n, seed, mismatches);
  return launch_status();
}

extern "C" moe_status_t moe_selftest_wait_timeout(uint64_t limit_ns, moe_stream_t stream) {
  MOE_CHECK_ARG(limit_ns >= 1000ull && limit_ns <= 10000000000ull);
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns);
  return launch_status();
}

extern "C" size_t moe_workspace_size_batched(int E, int max_tokens, int H, int I, const moe_quant_config* qc) {
  if (!qc || E < 1 || max_tokens < 1 || H <= 0 || I <= 0) return 0;
  return batched_layout(E, max_tokens, H, I, qc, gemm_grid()).total;
}

extern "C" moe_status_t moe_experts_batched(const void* a1q_b, const float* a1q_b_scale, const void* w13,
                                            const float* w13_scale, const void* w2, const float* w2_scale,
                                            const int32_t* expert_num_tokens, int E, int max_tokens, int H, int I,
                                            const moe_quant_config* qc, int activation, void* out_b, void* ws,
                                            size_t ws_bytes, moe_stream_t stream) {
  return experts_batched_run(a1q_b, a1q_b_scale, w13, w13_scale, w2, w2_scale, expert_num_tokens, E, max_tokens, H, I,
                             qc, activation, out_b, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}
