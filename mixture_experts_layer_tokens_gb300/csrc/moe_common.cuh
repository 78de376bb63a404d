// Shared device/host helpers of the fused-MoE library (sm_103a only).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a (Blackwell tcgen05/TMA); build with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace moe {

// ------------------------------------------------------------------ host helpers
#define MOE_CHECK_ARG(cond)                 \
  do {                                      \
    if (!(cond)) return MOE_ERR_INVALID_ARG; \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline moe_status_t launch_status() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int num_sms();                 // SM count of the current device (cached per device)
bool fits_int32(long long v);  // 0 <= v < 2^31

// Device status word: a wait that gives up records MOE_ERR_TIMEOUT, a kernel
// that meets an out-of-range index records MOE_ERR_INVALID_ARG.  Each
// translation unit has its own copy (no relocatable device code); the units
// that write it define a reader with MOE_DEFINE_STATUS_READER and
// moe_device_status combines them.
static __device__ int g_moe_status = 0;

#define MOE_DEFINE_STATUS_READER(fn)                                           \
  moe_status_t fn(int clear) {                                                 \
    int v = 0;                                                                 \
    if (cudaMemcpyFromSymbol(&v, g_moe_status, sizeof(int)) != cudaSuccess)    \
      return MOE_ERR_CUDA;                                                     \
    if (clear && v) {                                                          \
      const int z = 0;                                                         \
      if (cudaMemcpyToSymbol(g_moe_status, &z, sizeof(int)) != cudaSuccess)    \
        return MOE_ERR_CUDA;                                                   \
    }                                                                          \
    return (moe_status_t)v;                                                    \
  }

moe_status_t align_status(int clear);
moe_status_t experts_status(int clear);
moe_status_t prepare_status(int clear);
moe_status_t finalize_status(int clear);

__device__ __forceinline__ void record_status(int code) { atomicCAS(&g_moe_status, 0, code); }

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wall-clock limit of every device-side wait: long enough never to fire on a
// healthy run, short enough that a bug ends the kernel instead of hanging it.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void record_timeout() { record_status((int)MOE_ERR_TIMEOUT); }

__device__ __forceinline__ bool status_failed() {
  return *reinterpret_cast<volatile int*>(&g_moe_status) != 0;
}

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on the phase with parity `parity`.  Returns false (and records
// MOE_ERR_TIMEOUT) when the limit passes, or -- when `bail` -- as soon as any
// thread has recorded a failure.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, bool bail = true,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 255u) == 0) {
      if (bail && status_failed()) return false;
      if (global_ns() - t0 > limit_ns) {
        record_timeout();
        return false;
      }
    }
  }
}

// ---- cp.async (4-byte global -> shared copies; completion tracked by an mbarrier)
__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed (the
// barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---- TMA (bulk tensor copies, global -> shared, completion on an mbarrier)
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 3-D variant: box (x, y, z) at coordinates {x, y, z}.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Bring a tensor map's descriptor into the cache ahead of its first use.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T, both K-major, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with E4M3 inputs (kind::f8f6f4), fp32 accumulate.
__device__ __forceinline__ void mma_fp8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with NVFP4 inputs and block scaling (kind::mxf4nvf4, scale_vec::4X): packed
// E2M1 operands, one E4M3 scale per 16 K elements of every row of A and of B, read
// by the tensor core from tensor memory at sfa / sfb, fp32 accumulate.  The scales
// of one K = 64 step occupy 4 consecutive columns per 128 rows: the scale word
// (4 E4M3 codes, K groups 0-3 in bytes 0-3) of row l + 32 c sits in lane l of each
// 32-lane quarter, column c.
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of the block-scaled NVFP4 MMA: E2M1 A and B (format 1 of
// kind::mxf4nvf4), K-major, E4M3 scales (bit 23 clear), shape M x N, K = 64.
__host__ __device__ constexpr uint32_t make_idesc_nvf4(int M, int N) {
  return (1u << 7)                       // A format: E2M1
         | (1u << 10)                    // B format: E2M1
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// 32 lanes x 16 / 32 consecutive 32-bit columns from registers into tensor memory.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand stored in 128-byte
// swizzled rows (the layout a TMA load with SWIZZLE_128B writes): 8-row atoms
// of 1024 bytes, consecutive atoms 1024 bytes apart along M/N.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);  // start address, bits 0-13
  d |= (uint64_t)(16 >> 4) << 16;               // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset: next 8-row atom
  d |= (uint64_t)1 << 46;                       // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;                       // swizzle mode: 128-byte
  return d;
}

// Instruction descriptor: fp32 accumulator, K-major A and B, shape M x N.
// a_b_format: 1 = bf16 (kind::f16), 0 = E4M3 (kind::f8f6f4).
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_b_format, int M, int N) {
  return (1u << 4)                       // D format: fp32
         | (a_b_format << 7)             // A format
         | (a_b_format << 10)            // B format
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// 32 lanes x 32 consecutive fp32 columns from tensor memory into registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 64 consecutive fp32 columns.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
        "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
        "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
        "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// tmem_ld64 and the wait for it in one statement: the registers are defined only
// once the load has completed, so code using them can be scheduled freely after it.
__device__ __forceinline__ void tmem_ld64_wait(uint32_t taddr, float (&v)[64]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
        "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
        "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
        "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}


// ---- vector helpers of the quantisers
// 8 bf16 values (one 16-byte read-only load) as fp32
__device__ __forceinline__ void load_bf16x8(const void* p, float (&x)[8]) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16lo(w[i]);
    x[2 * i + 1] = bf16hi(w[i]);
  }
}

// The same through a coherent load (ld.global.cg): for rows that an earlier phase of
// the same kernel wrote, which the read-only path may not see.
__device__ __forceinline__ void load_bf16x8_cg(const void* p, float (&x)[8]) {
  const uint4 v = __ldcg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16lo(w[i]);
    x[2 * i + 1] = bf16hi(w[i]);
  }
}

__device__ __forceinline__ float amax8(const float (&x)[8]) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(x[i]));
  return a;
}

// x / s rounded to nearest (the IEEE quotient) for a divisor shared by many
// dividends, given rs = __frcp_rn(s), its correctly rounded reciprocal: q = RN(x rs) is
// within one ulp of x / s, the residual x - s q is exact in one fma, and RN(q + r rs) is
// then the correctly rounded quotient (P. Markstein, "IA-64 and Elementary Functions",
// 2000, the final correction step of division).  A zero quotient keeps the sign of x.
// Three operations per element against a full division each; the self-test
// moe_selftest_row_division compares it with __fdiv_rn bit for bit over the
// requantisation domain (divisors max(amax, 1e-10) / 448).
__device__ __forceinline__ float div_rn_by(float x, float s, float rs) {
  const float q = __fmul_rn(x, rs);
  const float r = __fmaf_rn(-q, s, x);
  return copysignf(__fmaf_rn(r, rs, q), x);
}

// 8 values -> 8 E4M3 codes with scale s: q = e4m3_rn_satfinite(fp32(x / s)), the quotient
// correctly rounded (div_rn_by)
__device__ __forceinline__ uint2 e4m3x8(const float (&x)[8], float s) {
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
  return make_uint2(packed[0], packed[1]);
}

// One NVFP4 group of 16 values with global scale g, every step in fp32:
// sf = e4m3_rn_satfinite(amax / (6 g)), q_i = e2m1_rn_satfinite(x_i / (sf g))
// (0 when sf g = 0).  Returns the 16 codes packed (element 2i in the low nibble
// of byte i) and writes the scale code.
__device__ __forceinline__ uint64_t nvfp4_group16(const float (&x)[16], float g, uint8_t& sf_code) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const __nv_fp8_storage_t sf8 = __nv_cvt_float_to_fp8(__fdiv_rn(amax, 6.0f * g), __NV_SATFINITE, __NV_E4M3);
  const float d = __half2float(__half(__nv_cvt_fp8_to_halfraw(sf8, __NV_E4M3))) * g;
  sf_code = (uint8_t)sf8;
  uint64_t q = 0;
  if (d > 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 r = make_float2(__fdiv_rn(x[2 * i], d), __fdiv_rn(x[2 * i + 1], d));
      q |= (uint64_t)__nv_cvt_float2_to_fp4x2(r, __NV_E2M1, cudaRoundNearest) << (8 * i);
    }
  }
  return q;
}

// Block-wide max of non-negative values over kThreads threads; every thread gets it.
template <int kThreads>
__device__ __forceinline__ float block_amax(float a) {
  __shared__ float red[kThreads / 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) a = fmaxf(a, red[w]);
  __syncthreads();
  return a;
}

}  // namespace moe
