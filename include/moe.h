/*
 * moe.h -- C ABI of the single-GPU fused mixture-of-experts layer (GB300, sm_103a).
 *
 * The layer is the modular no-DP/EP pipeline described by the pages:
 *
 *   moe_route    -> topk_ids, topk_weights
 *   moe_align    -> per-expert grouping of the (token, choice) slots
 *   moe_prepare  -> a1q (+ a1q_scale)                         ("prepare")
 *   moe_experts  -> fused_expert_output, unweighted rows      ("experts")
 *   moe_finalize -> output (+ residual_out)                   ("finalize")
 *
 * with the experts also in other forms: moe_experts_act (other activations),
 * moe_experts_multi (routed and shared experts in the same launches),
 * moe_prepare_nvfp4 / moe_experts_nvfp4 (every operand NVFP4); and the whole
 * bf16 step as one launch for decode-sized problems: moe_layer_fused.
 *
 * Sources: "[vLLM] MoE Oracle & Prepare/Finalize" blog, section "No DP/EP: the
 * simplest case" (prepare and finalize of MoEPrepareAndFinalizeNoDPEPModular);
 * "Fused MoE Kernel Features" (vLLM design doc), sections "Fused MoE Modular
 * All2All backends" and "Fused Experts Kernels"; "[flashinfer] MoE Finalize +
 * AllReduce fusion" page, introduction (finalize + shared row + residual +
 * RMSNorm + optional NVFP4 output).
 *
 * Conventions shared by every call
 *  - Every pointer argument is a DEVICE pointer on the current CUDA device,
 *    16-byte aligned, unless its comment says otherwise.  The caller owns and
 *    allocates every buffer, workspaces included; the library allocates no
 *    device memory.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and never synchronises (moe_device_status excepted).
 *  - Arguments are checked on the host before any launch; a bad argument
 *    returns an error status and launches nothing.  A launch failure returns
 *    MOE_ERR_CUDA.  No call aborts or throws.
 *  - Slot f = t * top_k + j names the j-th expert choice of token t.
 *  - Sizes are element counts; T (tokens) may be 0, in which case the call
 *    does nothing and returns MOE_OK.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad size or misaligned pointer   */
  MOE_ERR_UNSUPPORTED = 2,  /* valid request this library does not implement   */
  MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required      */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime/driver call or launch failed      */
  MOE_ERR_TIMEOUT = 5       /* a device-side wait gave up (see moe_device_status) */
} moe_status_t;

typedef enum {
  MOE_DT_BF16 = 0,
  MOE_DT_FP8_E4M3 = 1, /* OCP E4M3 ("e4m3fn"), saturating                    */
  MOE_DT_NVFP4 = 2,    /* E2M1 pairs + one E4M3 scale per 16 elements        */
  MOE_DT_FP32 = 3
} moe_dtype_t;

typedef enum {
  MOE_SCORING_SOFTMAX_RENORM = 0, /* softmax over the chosen top-k logits     */
  MOE_SCORING_SIGMOID = 1         /* top-1, weight = sigmoid(logit)           */
} moe_scoring_t;

/* Activation between the two expert GEMMs: the activation column of the
 * "Fused Experts Kernels" table (vLLM design doc), which names them without
 * formulas.  With [g | u] = x . w13^T (gate rows first):
 *   MOE_ACT_SILU         h = silu(g) * u,  silu(g) = g / (1 + exp(-g))
 *   MOE_ACT_GELU         h = gelu(g) * u,  gelu(g) = g/2 (1 + erf(g / sqrt 2))
 *   MOE_ACT_GELU_TANH    h = g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) * u
 *   MOE_ACT_SWIGLUOAI    the clamped SwiGLU of the gpt-oss models:
 *                        g' = min(g, 7), u' = clamp(u, -7, 7),
 *                        h = (u' + 1) * g' * sigmoid(1.702 g')
 *   MOE_ACT_SILU_NO_MUL  h = silu(g); w13 holds the I gate rows only
 *   MOE_ACT_GELU_NO_MUL  h = gelu(g); w13 holds the I gate rows only */
typedef enum {
  MOE_ACT_SILU = 0,
  MOE_ACT_GELU = 1,
  MOE_ACT_GELU_TANH = 2,
  MOE_ACT_SWIGLUOAI = 3,
  MOE_ACT_SILU_NO_MUL = 4,
  MOE_ACT_GELU_NO_MUL = 5
} moe_activation_t;

/* act_group values for the quantisation formats of the "Fused MoE Kernel
 * Features" tables besides G(128): "A" (per activation token) and "T" (per
 * tensor). */
#define MOE_GROUP_TOKEN (-1)  /* one scale per token over all H channels   */
#define MOE_GROUP_TENSOR (-2) /* one scale over the whole activation tensor */

/* Quantisation of the expert inputs and weights.
 *   bf16:  {MOE_DT_BF16, 0, MOE_DT_BF16, 0, 0}   -- "no quantisation type"
 *   fp8:   {MOE_DT_FP8_E4M3, 128, MOE_DT_FP8_E4M3, 128, 128}
 *          activations: one fp32 scale per token per 128 channels ("G(128)"),
 *          a1q_scale [T, H/128]; weights: one fp32 scale per 128x128 block.
 *   fp8 with act_group MOE_GROUP_TOKEN: a1q_scale [T] ("A");
 *            act_group MOE_GROUP_TENSOR: a1q_scale [1] ("T").
 *          Every scale is s = fp32(max(amax, 1e-10) / 448) over its group and
 *          q = e4m3_rn_satfinite(fp32(x / s)).  In moe_experts the
 *          intermediate h is quantised in the same format: G(128) from fp32 h;
 *          A and T from h stored in bf16 (T: one scale over every expert's rows).
 * Other combinations return MOE_ERR_UNSUPPORTED. */
typedef struct {
  moe_dtype_t act;
  int act_group;
  moe_dtype_t weight;
  int w_block_n;
  int w_block_k;
} moe_quant_config;

/* Rows per expert tile in the tile map that moe_experts consumes. */
#define MOE_BLOCK_M 128

/* ------------------------------------------------------------------ route
 * Router: top-k experts per token and their weights.  The pages take
 * topk_ids/topk_weights as inputs of prepare and finalize ("No DP/EP"
 * listing); the router is the plainest reading of them:
 *   MOE_SCORING_SOFTMAX_RENORM: the top_k largest fp32 logits, ordered larger
 *     first, equal logits to the lower expert index; weight_j =
 *     exp(l_j - l_max) / sum over the chosen i of exp(l_i - l_max).
 *   MOE_SCORING_SIGMOID (top_k must be 1): argmax (lower index on ties),
 *     weight = 1 / (1 + exp(-l)) -- the Llama-type router whose weight is
 *     applied on the input ("Fused MoE Kernel Features", All2All section).
 * logits [T, E] fp32 row-major; topk_ids [T, top_k] int32; topk_weights
 * [T, top_k] fp32.  1 <= E <= 1024, 1 <= top_k <= min(E, 32).  NaN logits rank
 * below every number. */
moe_status_t moe_route(const float *logits, int T, int E, int top_k, int scoring,
                       int32_t *topk_ids, float *topk_weights, moe_stream_t stream);

/* ------------------------------------------------------------------ align
 * Per-expert token alignment and permutation: the slots are sorted by the key
 * (expert id, slot f), which groups each expert's rows contiguously in
 * ascending slot order (deterministic).
 *   expert_offsets [E + 1] int32: exclusive prefix sum of the per-expert
 *                  counts; expert_offsets[E] = T * top_k.
 *   sorted_slot    [T * top_k] int32: sorted_slot[p] = f.
 *   inv_slot       [T * top_k] int32: inv_slot[sorted_slot[p]] = p (may be NULL).
 *   tile_map       [moe_tile_map_capacity(T * top_k, E, block_m)] pairs of
 *                  int32 (expert, first row p) for each block_m-row tile of
 *                  each expert, expert by expert; entries past num_tiles are
 *                  left untouched.
 *   num_tiles      [1] int32: number of valid tile_map entries.
 *   ws             scratch of moe_align_workspace_size(T, top_k, E) bytes.
 * topk_ids values must lie in [0, E); 1 <= E <= 1024; block_m >= 1
 * (moe_experts needs MOE_BLOCK_M). */
moe_status_t moe_align(const int32_t *topk_ids, int T, int top_k, int E, int block_m,
                       int32_t *expert_offsets, int32_t *sorted_slot, int32_t *inv_slot,
                       int32_t *tile_map, int32_t *num_tiles, void *ws, size_t ws_bytes,
                       moe_stream_t stream);
size_t moe_align_workspace_size(int T, int top_k, int E);
int moe_tile_map_capacity(int num_slots, int E, int block_m);

/* ------------------------------------------------------------------ align, no allocation
 * Not part of the method: the pages have no counterpart of this call.  It is
 * moe_align for callers that cannot allocate device memory at call time --
 * runtimes that plan every device buffer ahead and forbid allocation while
 * serving, or plugin-style hosts whose per-call hook may not allocate -- and so
 * cannot supply the `ws` scratch that moe_align needs.
 *
 * Same arguments, layouts and results as moe_align, minus ws/ws_bytes.  The
 * scratch is a fixed array of MOE_ALIGN_NOALLOC_SCRATCH_BYTES inside the
 * library (every GPU that loads the library holds it until the process exits);
 * a problem needing more (moe_align_workspace_size(T, top_k, E) larger than
 * that) is rejected with MOE_ERR_WORKSPACE before anything is launched.  The
 * call allocates nothing.
 *  - The first call in each CUDA context looks up the array's device address
 *    (cudaGetSymbolAddress) with that context current and caches it for the
 *    context: normally once per device (its primary context), and once more
 *    after a cudaDeviceReset or in a caller's own context, where the library's
 *    device code is loaded again at another address.  Make that first call
 *    before any stream capture in the context.
 *  - All calls share the one array and it keeps the last call's contents (each
 *    call writes every entry it later reads, so nothing needs clearing).  Calls
 *    whose work overlaps on the GPU -- on different streams, or from different
 *    host threads without ordering -- race on it: order them on one stream. */
#define MOE_ALIGN_NOALLOC_SCRATCH_BYTES (256 * 1024)
moe_status_t moe_align_noalloc(const int32_t *topk_ids, int T, int top_k, int E, int block_m,
                               int32_t *expert_offsets, int32_t *sorted_slot, int32_t *inv_slot,
                               int32_t *tile_map, int32_t *num_tiles, moe_stream_t stream);

/* ------------------------------------------------------------------ prepare
 * Prepare ("No DP/EP" listing): when apply_router_weight_on_input is set
 * (top_k must be 1) the input is first multiplied by the token's weight cast to
 * bf16, a1 <- bf16(a1 * bf16(w)); then it is quantised per qc->act:
 *   MOE_DT_BF16:     a1q [T, H] bf16 (a copy; when a1q == a1 and no weight is
 *                    applied nothing is launched -- the passthrough);
 *   MOE_DT_FP8_E4M3: a1q [T, H] E4M3 codes (uint8), a1q_scale [T, H/128] fp32:
 *                    s = fp32(max(amax, 1e-10f) / 448) per 128 channels,
 *                    q = e4m3_rn_satfinite(x / s) (IEEE fp32 division);
 *                    act_group MOE_GROUP_TOKEN: a1q_scale [T], one s per token;
 *                    MOE_GROUP_TENSOR: a1q_scale [1], one s for the tensor
 *                    (a1q_scale is also the reduction's scratch until the call's
 *                    last launch writes the scale).
 * a1 [T, H] bf16.  topk_weights [T, top_k] fp32 (read only with the weight
 * flag).  topk_ids is accepted for parity with the pages' signature and unused
 * (may be NULL).  H % 128 == 0 for fp8, H % 8 == 0 for bf16. */
moe_status_t moe_prepare(const void *a1, const float *topk_weights, const int32_t *topk_ids,
                         int T, int H, int top_k, int apply_router_weight_on_input,
                         const moe_quant_config *qc, void *a1q, float *a1q_scale,
                         moe_stream_t stream);

/* ------------------------------------------------------------------ experts
 * Grouped expert MLPs ("Fused Experts Kernels": two GEMMs with SiLU-and-mul
 * between them).  For every expert e and sorted row p in
 * [expert_offsets[e], expert_offsets[e+1]), with slot f = sorted_slot[p] and
 * token t = f / top_k:
 *   [g | u] = a1q[t] . w13[e]^T          (w13 [E, 2I, H]: rows 0..I-1 gate,
 *                                          rows I..2I-1 up; K-contiguous)
 *   h       = silu(g) * u                 (bf16, or E4M3 G(128) with fp8)
 *   fused_expert_output[f] = h . w2[e]^T  (w2 [E, H, I]; bf16 [T*top_k, H],
 *                                          token-major, unweighted)
 * Accumulation is fp32.  fp8: a1q E4M3 + a1q_scale in the qc->act_group
 * format (G(128) [T, H/128], A [T], T [1]); w13/w2 E4M3
 * with w13_scale [E, 2I/128, H/128] and w2_scale [E, H/128, I/128] fp32; each
 * 128-deep K block is scaled by a1q_scale * w_scale before it is added.
 * expert_offsets / sorted_slot / tile_map / num_tiles come from moe_align with
 * block_m = MOE_BLOCK_M.  sorted_slot may be NULL when E == 1 and top_k == 1
 * (identity permutation; tile_map and expert_offsets are still required).
 * ws: moe_workspace_size(...) bytes.  H % 128 == 0, I % 128 == 0. */
moe_status_t moe_experts(const void *a1q, const float *a1q_scale, const void *w13,
                         const float *w13_scale, const void *w2, const float *w2_scale,
                         const int32_t *expert_offsets, const int32_t *sorted_slot,
                         const int32_t *tile_map, const int32_t *num_tiles, int T, int H,
                         int I, int E, int top_k, const moe_quant_config *qc,
                         void *fused_expert_output, void *ws, size_t ws_bytes,
                         moe_stream_t stream);
/* moe_experts with another activation (a moe_activation_t); moe_experts is
 * this call with MOE_ACT_SILU.  For the *_NO_MUL activations w13 is [E, I, H]
 * (fp8: w13_scale [E, I/128, H/128]).  Same arguments, workspace and errors
 * otherwise; an unknown activation returns MOE_ERR_UNSUPPORTED. */
moe_status_t moe_experts_act(const void *a1q, const float *a1q_scale, const void *w13,
                             const float *w13_scale, const void *w2, const float *w2_scale,
                             const int32_t *expert_offsets, const int32_t *sorted_slot,
                             const int32_t *tile_map, const int32_t *num_tiles, int T, int H,
                             int I, int E, int top_k, const moe_quant_config *qc, int activation,
                             void *fused_expert_output, void *ws, size_t ws_bytes,
                             moe_stream_t stream);
size_t moe_workspace_size(int T, int H, int I, int E, int top_k, const moe_quant_config *qc);

/* Where moe_experts / moe_experts_act leave the intermediate h in their workspace
 * (it stays there until the workspace is used again), for inspection of the stage
 * between the two GEMMs.  Rows are the S = T * top_k sorted rows p (expert order):
 *   *h_offset       byte offset in ws of h [S, I]: bf16, or E4M3 codes for fp8;
 *   *h_scale_offset fp8 only (0 otherwise): byte offset of h's fp32 scales --
 *                   G(128): [I/128][*scale_stride], transposed (the scale of row p and
 *                   128-column group g at g * *scale_stride + p); "A" and "T": [S],
 *                   one per row (*scale_stride = 1; "T" repeats the tensor's scale);
 *   *scale_stride   as above (0 for bf16).
 * Same sizes and qc as the moe_experts call.  Returns MOE_ERR_INVALID_ARG on a bad
 * size or null pointer, MOE_ERR_UNSUPPORTED for a qc moe_experts rejects.  The
 * pages have no counterpart: it exposes a stage of the experts to the caller. */
moe_status_t moe_workspace_intermediate(int T, int H, int I, int E, int top_k, const moe_quant_config *qc,
                                        size_t *h_offset, size_t *h_scale_offset, int *scale_stride);

/* Several expert problems with the same hidden size H in the same two GEMM
 * launches -- typically a layer's routed experts and its shared expert (E = 1,
 * top_k = 1, sorted_slot NULL).  Not in the pages: their shared-expert row is a
 * separate MLP the finalize adds; computing both in one pass of launches saves
 * each GEMM's start-up and tail once (decode-sized layers spend a large share
 * of a GEMM there).  Each problem as for moe_experts_act, all with the same
 * activation and qc.  num_problems is 1 or 2; two problems need bf16 (qc) and
 * the same I (the second GEMM's depth), else MOE_ERR_UNSUPPORTED.  Problems
 * with no rows (T == 0) are skipped.  ws: moe_workspace_size_multi(...) bytes;
 * every output and error as for moe_experts. */
typedef struct {
  const void *a1q;
  const float *a1q_scale;
  const void *w13;
  const float *w13_scale;
  const void *w2;
  const float *w2_scale;
  const int32_t *expert_offsets;
  const int32_t *sorted_slot;
  const int32_t *tile_map;
  const int32_t *num_tiles;
  int T, I, E, top_k;
  void *fused_expert_output;
} moe_experts_problem;

moe_status_t moe_experts_multi(const moe_experts_problem *problems, int num_problems, int H,
                               const moe_quant_config *qc, int activation, void *ws,
                               size_t ws_bytes, moe_stream_t stream);
size_t moe_workspace_size_multi(const moe_experts_problem *problems, int num_problems, int H,
                                const moe_quant_config *qc);

/* ------------------------------------------------------------------ NVFP4 experts
 * The experts with every operand in NVFP4 ("Fused MoE Kernel Features", experts
 * table: nvfp4 is a quantisation type of the cutlass_fp4 and trtllm experts),
 * in the encoding of the finalize page's packed output: E2M1 codes in pairs
 * (element 2i in the low nibble), one E4M3 scale code per 16 consecutive
 * elements of a row, and one fp32 global scale g per tensor, value =
 * e2m1(q) * e4m3(sf) * g.  Quantising a row (prepare, the intermediate):
 *   sf = e4m3_rn_satfinite(fp32(amax16 / fp32(6 g))),
 *   q  = e2m1_rn_satfinite(fp32(x / fp32(e4m3(sf) * g)))   (q = 0 when that is 0).
 *
 * moe_prepare_nvfp4: a1 [T, H] bf16 (optionally first a1 <- bf16(a1 *
 *   bf16(w)) with the top-1 weight, as moe_prepare) -> a1q [T, H/2] codes,
 *   a1q_sf [T, H/16] scale codes, with the global scale *a1_gscale (device
 *   pointer, fp32, > 0).  H % 16 == 0; a1 and a1q 16-byte aligned.
 *
 * moe_experts_nvfp4: for every expert e and its sorted rows (as moe_experts):
 *   [g | u] = dequant(a1q[t]) . dequant(w13[e])^T    fp32 accumulation; the
 *            tensor core applies the E4M3 block scales, the product of the two
 *            global scales *a1_gscale * w13_gscale[e] multiplies the sums
 *   h      = act(g, u) stored bf16, then quantised to NVFP4 with *h_gscale
 *   fused_expert_output[f] = dequant(h) . dequant(w2[e])^T   (bf16 [T*top_k, H],
 *            token-major, unweighted)
 * w13 [E, 2I, H/2] codes with w13_sf [E, 2I, H/16] (rows 0..I-1 gate, I..2I-1
 * up; the *_NO_MUL activations: [E, I, H/2] and [E, I, H/16]); w2 [E, H, I/2]
 * with w2_sf [E, H, I/16]; w13_gscale, w2_gscale [E] fp32; a1_gscale, h_gscale
 * [1] fp32 (all device pointers).  expert_offsets / sorted_slot / tile_map /
 * num_tiles as for moe_experts (sorted_slot NULL only when E == 1 and top_k ==
 * 1).  H % 256 == 0, I % 256 == 0; every code, scale and output pointer 16-byte
 * aligned.  ws: moe_workspace_size_nvfp4(...) bytes (MOE_ERR_WORKSPACE when
 * smaller); an unknown activation returns MOE_ERR_UNSUPPORTED.  The caller owns
 * every buffer; nothing is allocated. */
moe_status_t moe_prepare_nvfp4(const void *a1, const float *topk_weights, int T, int H, int top_k,
                               int apply_router_weight_on_input, const float *a1_gscale, void *a1q,
                               void *a1q_sf, moe_stream_t stream);
moe_status_t moe_experts_nvfp4(const void *a1q, const void *a1q_sf, const float *a1_gscale,
                               const void *w13, const void *w13_sf, const float *w13_gscale,
                               const void *w2, const void *w2_sf, const float *w2_gscale,
                               const float *h_gscale, const int32_t *expert_offsets,
                               const int32_t *sorted_slot, const int32_t *tile_map,
                               const int32_t *num_tiles, int T, int H, int I, int E, int top_k,
                               int activation, void *fused_expert_output, void *ws, size_t ws_bytes,
                               moe_stream_t stream);
size_t moe_workspace_size_nvfp4(int T, int H, int I, int E, int top_k);
/* Where moe_experts_nvfp4 leaves the intermediate in its workspace: byte offsets of
 * the bf16 h [S, I] that the first GEMM writes, and of its NVFP4 codes [S, I/2] and
 * scale codes [S, I/16] that the second GEMM reads (S = T * top_k sorted rows).
 * H % 256 == 0 and I % 256 == 0, else MOE_ERR_INVALID_ARG. */
moe_status_t moe_workspace_intermediate_nvfp4(int T, int H, int I, int E, int top_k, size_t *hb_offset,
                                              size_t *hq_offset, size_t *hsf_offset);

/* ------------------------------------------------------------------ batched activation format
 * The "batched" format of the prepare output ("Fused MoE Kernel Features", section "Fused MoE
 * Modular All2All backends": a prepare returns its activations in the standard or the batched
 * format and the finalize takes that format back to standard; "Fused Experts Kernels" lists
 * batched entry points).  The pages leave the layout to another document; the reading here:
 * one slab per expert, [E, max_tokens, H]: expert e's slab holds, in ascending slot order, the
 * prepared rows of the tokens that chose e, and expert_num_tokens[e] counts them.  Rows past a
 * count are neither written nor read.
 *
 * moe_prepare_batched: moe_prepare (same qc, same weight on the input) of every token, then
 *   token t's prepared row copied to the slab of each expert it chose.  expert_offsets and
 *   sorted_slot are moe_align's (they give each expert's slots in ascending order).  Outputs:
 *   a1q_b [E, max_tokens, H] (bf16 or E4M3 codes); a1q_b_scale: G(128) [E, max_tokens, H/128],
 *   "A" [E, max_tokens], "T" [1] (fp32; unused for bf16, may be NULL); expert_num_tokens [E]
 *   int32 (each count capped at max_tokens).  A slot past max_tokens in its expert's slab is
 *   left out and MOE_ERR_INVALID_ARG is recorded in the device status word (moe_device_status);
 *   nothing is written out of bounds.  ws: moe_prepare_batched_workspace_size(T, H, qc) bytes
 *   (bf16 without the weight on the input needs none: the rows come from a1 itself).
 * moe_experts_batched: the experts of moe_experts_act on the slabs: for every expert e and row
 *   m < expert_num_tokens[e] (taken as min(max(count, 0), max_tokens)), out_b[e, m] =
 *   expert_e(a1q_b[e, m]); out_b [E, max_tokens, H] bf16, unweighted; other rows untouched.
 *   Same weights, qc, activations and intermediate as moe_experts_act.  ws:
 *   moe_workspace_size_batched(E, max_tokens, H, I, qc) bytes.  H % 128 == 0, I % 128 == 0.
 * moe_finalize_batched: moe_finalize reading the expert row of slot f = t * top_k + j from
 *   expert_output_b [E, max_tokens, H] at (e = topk_ids[f], inv_slot[f] - expert_offsets[e])
 *   (moe_align's inv_slot and expert_offsets); every other argument, output and check as for
 *   moe_finalize. */
size_t moe_prepare_batched_workspace_size(int T, int H, const moe_quant_config *qc);
moe_status_t moe_prepare_batched(const void *a1, const float *topk_weights, const int32_t *expert_offsets,
                                 const int32_t *sorted_slot, int T, int H, int top_k, int E, int max_tokens,
                                 int apply_router_weight_on_input, const moe_quant_config *qc, void *a1q_b,
                                 float *a1q_b_scale, int32_t *expert_num_tokens, void *ws, size_t ws_bytes,
                                 moe_stream_t stream);
size_t moe_workspace_size_batched(int E, int max_tokens, int H, int I, const moe_quant_config *qc);
moe_status_t moe_experts_batched(const void *a1q_b, const float *a1q_b_scale, const void *w13,
                                 const float *w13_scale, const void *w2, const float *w2_scale,
                                 const int32_t *expert_num_tokens, int E, int max_tokens, int H, int I,
                                 const moe_quant_config *qc, int activation, void *out_b, void *ws,
                                 size_t ws_bytes, moe_stream_t stream);
moe_status_t moe_finalize_batched(void *output, const void *expert_output_b, int max_tokens,
                                  const float *topk_weights, const int32_t *topk_ids, const int32_t *inv_slot,
                                  const int32_t *expert_offsets, const void *shared, const void *residual,
                                  const void *rms_weight, float eps, int T, int H, int top_k,
                                  int apply_router_weight_on_input, moe_dtype_t out_dtype, uint8_t *out_scale,
                                  float out_global_scale, void *residual_out, moe_stream_t stream);

/* ------------------------------------------------------------------ single-launch layer
 * The whole bf16 layer step in one cooperative kernel launch -- the monolithic form of
 * the experts ("[vLLM] MoE Oracle & Prepare/Finalize", section "Modular vs
 * Monolithic": one kernel from the router logits to the layer output) -- for
 * decode-sized problems.  Its phases, separated by grid-wide barriers, compute what the
 * separate calls do: moe_route (scoring as there), moe_align (the same order),
 * prepare (bf16; a1 <- bf16(a1 * bf16(w)) with apply_router_weight_on_input, top_k 1),
 * the experts with SiLU-and-mul (the shared expert, when given, in the same GEMM units
 * on the unweighted a1), and moe_finalize's sum (weights skipped with the weight on the
 * input) + shared row + residual, RMSNorm when rms_weight is given, bf16 output.
 * logits [T, E] fp32; a1 [T, H] bf16; w13 [E, 2I, H], w2 [E, H, I] bf16; shared_w13
 * [2I, H] and shared_w2 [H, I] bf16, both or neither; residual [T, H] and rms_weight
 * [H] bf16 or NULL; topk_ids / topk_weights [T, top_k] are written as by moe_route;
 * output [T, H] bf16.  Limits: T * top_k <= 2048, E <= 256, H and I multiples of 128,
 * H <= 12288; beyond them, or on a device without cooperative launch,
 * MOE_ERR_UNSUPPORTED.  ws: moe_layer_fused_workspace_size(...) bytes, caller-owned;
 * every wait (the grid barriers included) gives up as described under "status". */
moe_status_t moe_layer_fused(const float *logits, const void *a1, int T, int H, int I, int E, int top_k,
                             int scoring, int apply_router_weight_on_input, const void *w13, const void *w2,
                             const void *shared_w13, const void *shared_w2, const void *residual,
                             const void *rms_weight, float eps, int32_t *topk_ids, float *topk_weights,
                             void *output, void *ws, size_t ws_bytes, moe_stream_t stream);
size_t moe_layer_fused_workspace_size(int T, int H, int I, int E, int top_k, int has_shared);

/* ------------------------------------------------------------------ finalize
 * Finalize: the top-k weight-and-reduce of the "No DP/EP" listing followed by
 * the single-GPU part of the flashinfer finalize fusion (introduction of its
 * page, all-reduce removed):
 *   o_t = sum_j w_tj * y[t*top_k + j]   (w_tj = 1 when the weights were
 *                                         applied on the input)
 *         + shared_t + residual_t        (each optional: NULL = absent)
 *   residual_out_t = bf16(o_t)           (optional, NULL = not written)
 *   o_t <- o_t * rsqrt(mean_h(o_t^2) + eps) * rms_weight  (when rms_weight)
 * Sums in fp32.  Output per out_dtype:
 *   MOE_DT_BF16:  output [T, H] bf16;
 *   MOE_DT_FP32:  output [T, H] fp32;
 *   MOE_DT_NVFP4: output [T, H/2] uint8, element 2i in the low nibble, and
 *                 out_scale [T, H/16] E4M3 codes: per 16 elements
 *                 sf = e4m3(amax / (6 g)), q = e2m1(x / (sf g)), g =
 *                 out_global_scale > 0.
 * fused_expert_output [T*top_k, H] bf16; topk_weights [T, top_k] fp32;
 * shared, residual, residual_out [T, H] bf16; rms_weight [H] bf16.  residual_out
 * may be residual itself (the sum is then written over the residual, in place);
 * any other overlap between inputs and outputs is not allowed.  topk_ids
 * is accepted for parity with the pages' signature and unused (may be NULL).
 * H % 8 == 0 (H % 16 == 0 for NVFP4), 1 <= top_k <= 32. */
moe_status_t moe_finalize(void *output, const void *fused_expert_output, const float *topk_weights,
                          const int32_t *topk_ids, const void *shared, const void *residual,
                          const void *rms_weight, float eps, int T, int H, int top_k,
                          int apply_router_weight_on_input, moe_dtype_t out_dtype,
                          uint8_t *out_scale, float out_global_scale, void *residual_out,
                          moe_stream_t stream);

/* ------------------------------------------------------------------ status
 * Every device-side wait in the library's kernels gives up after about two
 * seconds, records MOE_ERR_TIMEOUT in a device status word and lets the
 * kernel return.  moe_device_status synchronises the current device, returns
 * the recorded status (MOE_OK when none) and clears it when `clear` != 0. */
moe_status_t moe_device_status(int clear);

/* Self-test of that failure path (the pages have no counterpart; it is not a step of the
 * layer): launches one thread that waits, with the same bounded wait the GEMM kernels
 * use, on a barrier no thread ever arrives on, giving up after limit_ns nanoseconds
 * (1e3 .. 1e10) instead of the usual two seconds.  The wait runs out, MOE_ERR_TIMEOUT is
 * recorded in the device status word and the kernel returns normally: the context stays
 * usable, moe_device_status reports the timeout (and clears it when asked).  Nothing
 * faults, traps or hangs.  Asynchronous on stream; MOE_ERR_INVALID_ARG for a limit out of
 * range. */
moe_status_t moe_selftest_wait_timeout(uint64_t limit_ns, moe_stream_t stream);

/* Self-test of the division the fp8 GEMM1 epilogue uses to requantise h (each element
 * divided by its row group's scale s = max(amax, 1e-10) / 448, "[vLLM] MoE Oracle &
 * Prepare/Finalize", the G(128) quantisation): the correctly rounded quotient from the
 * divisor's correctly rounded reciprocal and one fma correction, compared bit for bit with
 * the IEEE division on n pseudo-random (dividend, divisor) pairs of that domain drawn
 * from seed on the device.  *mismatches (device memory, zeroed by the caller) receives the
 * count of differing results.  Asynchronous on stream; MOE_ERR_INVALID_ARG for n < 0 or a
 * NULL counter. */
moe_status_t moe_selftest_row_division(long long n, uint32_t seed, unsigned long long *mismatches,
                                       moe_stream_t stream);
const char *moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
