// moe_align: per-expert grouping of the token slots (alignment + permutation).
//
// The slots f = t*k + j are sorted by the key (expert, f): each expert's rows
// become contiguous, in ascending slot order, so the permutation is exact and
// deterministic.  expert_offsets is the unpadded exclusive prefix sum of the
// per-expert counts; the tile map lists the block_m-row tiles of each expert.
//
// Up to kChunk slots, one launch (align_small_kernel: one block counts, scans
// and scatters with the same steps); beyond that three launches over chunks of
// kChunk slots:
//   1. count:   per-chunk histogram of expert ids              -> ws[chunk][E]
//   2. scan:    one block turns the histograms into expert offsets, per-chunk
//               bases (in place) and the tile map
//   3. scatter: each chunk ranks its slots stably and writes sorted_slot and
//               inv_slot.  A chunk is walked in rounds of 256 slots; inside a
//               round each warp ranks its 32 slots with __match_any_sync and
//               publishes per-expert counts tagged with the round number, so
//               later warps add the counts of earlier ones without clearing
//               any table.
// No result depends on the order in which atomics land.
#include <mutex>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;         // threads of the count/scatter blocks
constexpr int kRounds = 8;            // rounds of kThreads slots per chunk
constexpr int kChunk = kThreads * kRounds;
constexpr int kWarps = kThreads / 32;
constexpr int kScanThreads = 1024;    // also the largest supported E
constexpr int kBatch = 16;            // chunk histograms loaded per batch in the scan

__global__ void __launch_bounds__(kThreads)
    align_count_kernel(const int32_t* __restrict__ ids, int S, int E, int32_t* __restrict__ hist) {
  extern __shared__ int32_t h[];
  for (int e = threadIdx.x; e < E; e += kThreads) h[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kChunk;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int f = base + r * kThreads + threadIdx.x;
    if (f < S) {
      const int e = __ldg(ids + f);
      if ((unsigned)e < (unsigned)E)
        atomicAdd(&h[e], 1);
      else
        record_status((int)MOE_ERR_INVALID_ARG);  // the slot is left out of the permutation
    }
  }
  __syncthreads();
  int32_t* out = hist + (size_t)blockIdx.x * E;
  for (int e = threadIdx.x; e < E; e += kThreads) out[e] = h[e];
}

// Block-wide exclusive scan of one int per thread (kScanThreads threads).
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
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
    if (lane == 31) *total = wx;
  }
  __syncthreads();
  const int r = warp_tot[warp] + x - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kScanThreads)
    align_scan_kernel(int32_t* __restrict__ hist, int nchunks, int E, int block_m, int32_t* __restrict__ offsets,
                      int32_t* __restrict__ tile_map, int32_t* __restrict__ num_tiles) {
  __shared__ int warp_tot[32];
  __shared__ int total_rows, total_tiles;
  const int e = threadIdx.x;
  int count = 0;
  if (e < E) {
    for (int c0 = 0; c0 < nchunks; c0 += kBatch) {
      int n[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) n[u] = c0 + u < nchunks ? hist[(size_t)(c0 + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) count += n[u];
    }
  }
  const int off = block_exclusive_scan(count, warp_tot, &total_rows);
  const int ntile = e < E ? (count + block_m - 1) / block_m : 0;
  const int tstart = block_exclusive_scan(ntile, warp_tot, &total_tiles);
  if (e < E) {
    offsets[e] = off;
    int run = off;  // base of expert e's rows in each chunk, in chunk order
    for (int c0 = 0; c0 < nchunks; c0 += kBatch) {
      int n[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) n[u] = c0 + u < nchunks ? hist[(size_t)(c0 + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (c0 + u < nchunks) hist[(size_t)(c0 + u) * E + e] = run;
        run += n[u];
      }
    }
    for (int i = 0; i < ntile; ++i) {
      tile_map[2 * (tstart + i)] = e;
      tile_map[2 * (tstart + i) + 1] = off + i * block_m;
    }
  }
  if (threadIdx.x == 0) {
    offsets[E] = total_rows;
    *num_tiles = total_tiles;
  }
}

__global__ void __launch_bounds__(kThreads)
    align_scatter_kernel(const int32_t* __restrict__ ids, int S, int E, const int32_t* __restrict__ base,
                         int32_t* __restrict__ sorted_slot, int32_t* __restrict__ inv_slot) {
  extern __shared__ int32_t sm[];
  int32_t* running = sm;       // [E] rows of each expert placed by earlier rounds
  int32_t* wcnt = sm + E;      // [kWarps][E] (round + 1) << 16 | count of the expert in that warp
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < E; i += kThreads) running[i] = __ldg(base + (size_t)blockIdx.x * E + i);
  for (int i = threadIdx.x; i < kWarps * E; i += kThreads) wcnt[i] = 0;
  __syncthreads();
  const int chunk0 = blockIdx.x * kChunk;
  for (int r = 0; r < kRounds; ++r) {
    const int f = chunk0 + r * kThreads + threadIdx.x;
    int e = f < S ? __ldg(ids + f) : -1;
    const bool valid = (unsigned)e < (unsigned)E;
    if (!valid) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int in_warp = __popc(peers & ((1u << lane) - 1u));
    const bool leader = in_warp == 0;
    const int tag = (r + 1) << 16;
    if (valid && leader) wcnt[warp * E + e] = tag | __popc(peers);
    __syncthreads();
    int before = 0, after = 0;
    if (valid) {
      for (int w = 0; w < kWarps; ++w) {
        const int v = wcnt[w * E + e];
        const int c = (v & 0xFFFF0000) == tag ? (v & 0xFFFF) : 0;
        if (w < warp) before += c;
        if (w > warp) after += c;
      }
      const int p = running[e] + before + in_warp;
      sorted_slot[p] = f;
      if (inv_slot) inv_slot[f] = p;
    }
    __syncthreads();
    // the last warp holding expert e this round advances its running count
    if (valid && leader && after == 0) running[e] += before + __popc(peers);
    __syncthreads();
  }
}

// Small problems (S <= kChunk): count, scan and stable scatter in one block of
// kScanThreads threads, the scatter in rounds of kScanThreads slots ranked as in
// align_scatter_kernel.  Dynamic shared memory: (1 + 32) * E ints.
__global__ void __launch_bounds__(kScanThreads)
    align_small_kernel(const int32_t* __restrict__ ids, int S, int E, int block_m, int32_t* __restrict__ offsets,
                       int32_t* __restrict__ tile_map, int32_t* __restrict__ num_tiles,
                       int32_t* __restrict__ sorted_slot, int32_t* __restrict__ inv_slot) {
  constexpr int kW = kScanThreads / 32;
  extern __shared__ int32_t sm[];
  int32_t* h = sm;         // [E] counts, then the running row of each expert
  int32_t* wcnt = sm + E;  // [kW][E] (round + 1) << 16 | count of the expert in that warp
  __shared__ int warp_tot[32];
  __shared__ int total_rows, total_tiles;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < E; i += kScanThreads) h[i] = 0;
  for (int i = threadIdx.x; i < kW * E; i += kScanThreads) wcnt[i] = 0;
  __syncthreads();
  for (int f = threadIdx.x; f < S; f += kScanThreads) {
    const int e = __ldg(ids + f);
    if ((unsigned)e < (unsigned)E)
      atomicAdd(&h[e], 1);
    else
      record_status((int)MOE_ERR_INVALID_ARG);  // the slot is left out of the permutation
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int count = e < E ? h[e] : 0;
  const int off = block_exclusive_scan(count, warp_tot, &total_rows);
  const int ntile = e < E ? (count + block_m - 1) / block_m : 0;
  const int tstart = block_exclusive_scan(ntile, warp_tot, &total_tiles);
  if (e < E) {
    offsets[e] = off;
    h[e] = off;
    for (int i = 0; i < ntile; ++i) {
      tile_map[2 * (tstart + i)] = e;
      tile_map[2 * (tstart + i) + 1] = off + i * block_m;
    }
  }
  if (threadIdx.x == 0) {
    offsets[E] = total_rows;
    *num_tiles = total_tiles;
  }
  __syncthreads();
  for (int r = 0; r * kScanThreads < S; ++r) {
    const int f = r * kScanThreads + threadIdx.x;
    int x = f < S ? __ldg(ids + f) : -1;
    const bool valid = (unsigned)x < (unsigned)E;
    if (!valid) x = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, x);
    const int in_warp = __popc(peers & ((1u << lane) - 1u));
    const bool leader = in_warp == 0;
    const int tag = (r + 1) << 16;
    if (valid && leader) wcnt[warp * E + x] = tag | __popc(peers);
    __syncthreads();
    int before = 0, after = 0;
    if (valid) {
      for (int w = 0; w < kW; ++w) {
        const int v = wcnt[w * E + x];
        const int c = (v & 0xFFFF0000) == tag ? (v & 0xFFFF) : 0;
        if (w < warp) before += c;
        if (w > warp) after += c;
      }
      const int p = h[x] + before + in_warp;
      sorted_slot[p] = f;
      if (inv_slot) inv_slot[f] = p;
    }
    __syncthreads();
    if (valid && leader && after == 0) h[x] += before + __popc(peers);
    __syncthreads();
  }
}

}  // namespace

MOE_DEFINE_STATUS_READER(align_status)

}  // namespace moe

using namespace moe;

extern "C" size_t moe_align_workspace_size(int T, int top_k, int E) {
  if (T < 0 || top_k < 1 || E < 1) return 0;
  const long long S = (long long)T * top_k;
  const long long nchunks = (S + kChunk - 1) / kChunk;
  return (size_t)((nchunks > 0 ? nchunks : 1) * E * sizeof(int32_t));
}

extern "C" int moe_tile_map_capacity(int num_slots, int E, int block_m) {
  if (num_slots < 0 || E < 1 || block_m < 1) return -1;
  if (num_slots == 0) return 0;
  const long long cap = ((long long)num_slots + (long long)E * (block_m - 1)) / block_m;
  return (int)(cap < num_slots ? cap : num_slots);
}

extern "C" moe_status_t moe_align(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                                  int32_t* expert_offsets, int32_t* sorted_slot, int32_t* inv_slot,
                                  int32_t* tile_map, int32_t* num_tiles, void* ws, size_t ws_bytes,
                                  moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && top_k >= 1 && E >= 1 && E <= kScanThreads && block_m >= 1);
  MOE_CHECK_ARG(fits_int32((long long)T * top_k));
  MOE_CHECK_ARG(expert_offsets && tile_map && num_tiles);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int S = T * top_k;
  if (S > 0) {
    MOE_CHECK_ARG(topk_ids && sorted_slot);
    if (!ws || ws_bytes < moe_align_workspace_size(T, top_k, E)) return MOE_ERR_WORKSPACE;
  }
  const int nchunks = (S + kChunk - 1) / kChunk;
  if (nchunks == 1) {
    const size_t smem = (size_t)(1 + kScanThreads / 32) * E * sizeof(int32_t);  // <= 132 KB at E = 1024
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
      if (cudaFuncSetAttribute(align_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)((1 + kScanThreads / 32) * kScanThreads * sizeof(int32_t))) != cudaSuccess)
        return MOE_ERR_CUDA;
      configured[dev] = 1;
    }
    align_small_kernel<<<1, kScanThreads, smem, s>>>(topk_ids, S, E, block_m, expert_offsets, tile_map, num_tiles,
                                                     sorted_slot, inv_slot);
    return launch_status();
  }
  int32_t* hist = static_cast<int32_t*>(ws);
  if (nchunks > 0) align_count_kernel<<<nchunks, kThreads, E * sizeof(int32_t), s>>>(topk_ids, S, E, hist);
  align_scan_kernel<<<1, kScanThreads, 0, s>>>(hist, nchunks, E, block_m, expert_offsets, tile_map, num_tiles);
  if (nchunks > 0) {
    const size_t smem = (size_t)(1 + kWarps) * E * sizeof(int32_t);  // <= 36 KB at E = 1024
    align_scatter_kernel<<<nchunks, kThreads, smem, s>>>(topk_ids, S, E, hist, sorted_slot, inv_slot);
  }
  return launch_status();
}

// ------------------------------------------------------------------ align without allocation
// Scratch of moe_align_noalloc: a file-scope device array shared by every call.
// On the host this name is only a stand-in for the symbol, not a device
// address: host code passes kernels the address looked up below, once per
// CUDA context (normally once per device).
static __device__ __align__(256) int32_t g_align_scratch[MOE_ALIGN_NOALLOC_SCRATCH_BYTES / sizeof(int32_t)];

namespace {
// The array's device address belongs to the module as loaded in one CUDA
// context: a cudaDeviceReset, or a caller's own (non-primary) context, loads
// the module again at another address.  So the looked-up address is cached per
// context, keyed on the context's unique id (cuCtxGetId: never reused within
// the process, unlike the context handle).
constexpr int kCacheEntries = 64;
struct ScratchEntry {
  unsigned long long ctx_id;
  int32_t* ptr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch_cache[kCacheEntries];
int g_scratch_used = 0;

using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

template <class F>
F driver_fn(const char* name, int version) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(fn);
}

// Unique id of the current context, or 0 when none is current yet.
bool current_ctx_id(unsigned long long* id) {
  static PfnCtxGetCurrent get_current = driver_fn<PfnCtxGetCurrent>("cuCtxGetCurrent", 4000);
  static PfnCtxGetId get_id = driver_fn<PfnCtxGetId>("cuCtxGetId", 12000);
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  return !ctx || get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_align_scratch in the current context (the current
// device's primary context unless the caller made another current), looked up
// with cudaGetSymbolAddress on the first call in that context and cached.
moe_status_t scratch_on_current_device(int32_t** out) {
  unsigned long long id = 0;
  if (!current_ctx_id(&id)) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (id) {
    for (int i = 0; i < g_scratch_used; ++i)
      if (g_scratch_cache[i].ctx_id == id) {
        *out = g_scratch_cache[i].ptr;
        return MOE_OK;
      }
  }
  // (with no context current yet, the lookup itself makes the device's primary
  // context current; its id is read afterwards)
  int32_t* p = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_align_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
  if (!id && (!current_ctx_id(&id) || !id)) return MOE_ERR_CUDA;
  const int slot = g_scratch_used < kCacheEntries ? g_scratch_used++ : (int)(id % kCacheEntries);
  g_scratch_cache[slot] = {id, p};
  *out = p;
  return MOE_OK;
}
}  // namespace

extern "C" moe_status_t moe_align_noalloc(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                                          int32_t* expert_offsets, int32_t* sorted_slot, int32_t* inv_slot,
                                          int32_t* tile_map, int32_t* num_tiles, moe_stream_t stream) {
  MOE_CHECK_ARG(T >= 0 && top_k >= 1 && E >= 1 && E <= kScanThreads && block_m >= 1);
  MOE_CHECK_ARG(fits_int32((long long)T * top_k));
  MOE_CHECK_ARG(expert_offsets && tile_map && num_tiles);
  const int S = T * top_k;
  if (S > 0) MOE_CHECK_ARG(topk_ids && sorted_slot);
  if (moe_align_workspace_size(T, top_k, E) > (size_t)MOE_ALIGN_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  int32_t* hist = nullptr;
  const moe_status_t st = scratch_on_current_device(&hist);
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int nchunks = (S + kChunk - 1) / kChunk;
  if (nchunks > 0) align_count_kernel<<<nchunks, kThreads, E * sizeof(int32_t), s>>>(topk_ids, S, E, hist);
  align_scan_kernel<<<1, kScanThreads, 0, s>>>(hist, nchunks, E, block_m, expert_offsets, tile_map, num_tiles);
  if (nchunks > 0) {
    const size_t smem = (size_t)(1 + kWarps) * E * sizeof(int32_t);
    align_scatter_kernel<<<nchunks, kThreads, smem, s>>>(topk_ids, S, E, hist, sorted_slot, inv_slot);
  }
  return launch_status();
}
