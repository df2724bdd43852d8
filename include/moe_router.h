/*
 * moe_router.h — fused Mixture-of-Experts router for NVIDIA GB300 (sm_103a).
 *
 * C ABI over caller-owned device memory.  The core operations are the two
 * fused router ops of NVIDIA TransformerEngine PR #3012 "[Common] Optimize
 * fused router forward/backward kernels" (Summary: fused_topk_with_score_
 * function and fused_score_for_moe_aux_loss, each with a forward and a
 * backward).  Around them: the router with compact [T, K] outputs, the
 * (expert, token)-sorted expert maps and the one-launch decode router with
 * maps, and the load-balancing aux loss (each documented below with the page
 * it follows).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every [T, E] tensor is dense row-major with row stride E elements, in
 *   device memory owned by the caller.  Nothing is allocated, freed or
 *   synchronised here: each call validates its arguments on the host,
 *   enqueues its work on `stream` (one kernel for the router ops; the calls
 *   with a workspace say what they enqueue) and returns.  Kernels are
 *   launched with programmatic dependent launch (each waits for the previous
 *   kernel in the stream before touching memory; MOE_ROUTER_PDL=0 disables
 *   it).  Above 512 experts, a forward with more rows than the GPU holds
 *   warps at once launches one one-warp block per row whose running warps
 *   take over the rows of blocks not yet started (cluster launch control);
 *   a compact forward of fp32 rows above 1024 experts with no dense output
 *   keeps one row buffer per warp instead of two in that launch.  The
 *   results are those of the persistent launch, bit for bit
 *   (MOE_ROUTER_STEAL=0 keeps the persistent launch).
 * - `dtype` is the type of the logits and of the tensors that follow it
 *   (probs, grad_probs, grad_logits): MR_F32 (float) or MR_BF16
 *   (__nv_bfloat16).  Scores, intermediates, grad_scores and the expert bias
 *   are always float; routing maps are one byte per element, 0 or 1.
 * - All arithmetic is fp32 (bf16 inputs are widened exactly); bf16 outputs are
 *   rounded to nearest-even once, at the store.
 * - Ties in the top-K choice go to the lower expert index (and, for grouped
 *   routing, to the lower group index); -0.0 and +0.0 are equal.
 * - Inputs must be finite; NaN or Inf logits give unspecified (but in-bounds)
 *   results.
 * - T == 0 is a successful no-op once the other arguments have been checked;
 *   tensor pointers may then be NULL (empty tensors have no storage).
 * - Pointers need no particular alignment; rows that are not 16-byte aligned
 *   take a slower element-wise path.
 * - Return value: MR_OK (0) or a negative mr_status.  On an argument error
 *   nothing is written and nothing is enqueued.  MR_ERR_CUDA reports a failed
 *   launch (cudaGetLastError); kernels already enqueued are not undone.
 * - The buffers must live on the calling thread's current CUDA device.
 * - Calls are thread-safe with respect to each other except
 *   moe_router_force_path and moe_router_force_fwd_lanes, which set
 *   process-wide state.
 */
#ifndef MOE_ROUTER_H
#define MOE_ROUTER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MR_API __attribute__((visibility("default")))
#else
#define MR_API
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* mr_stream_t;

/*
 * MR_SOFTMAX_POST is the post-softmax router (TransformerEngine PR #3012's
 * review names the ScoreFunc x use_pre_softmax combinations; onnxruntime PR
 * #33366 calls it normalize_routing_weights): it selects and scores like
 * MR_SOFTMAX, and its probs are the softmax of the K selected logits.  The
 * aux-score calls take MR_SOFTMAX and MR_SIGMOID only.
 */
typedef enum { MR_SOFTMAX = 0, MR_SIGMOID = 1, MR_SOFTMAX_POST = 2 } mr_score_func;
typedef enum { MR_F32 = 0, MR_BF16 = 1 } mr_dtype;

typedef enum {
  MR_OK = 0,
  MR_ERR_INVALID = -1,      /* an argument breaks the rules stated per call */
  MR_ERR_UNSUPPORTED = -2,  /* valid, but beyond this build's limits below   */
  MR_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed          */
} mr_status;

/* Limits of this build (MR_ERR_UNSUPPORTED beyond them). */
#define MR_MAX_EXPERTS 2304
#define MR_MAX_TOPK 36
#define MR_MAX_GROUPS 32

/*
 * router_topk_fwd — score, select and emit the top-K experts of each token.
 *
 * Source: TransformerEngine PR #3012, Summary and Performance (the forward
 * reads logits [T,E] and writes probs [T,E] in the logits dtype, the routing
 * map [T,E] as one byte per element and the fp32 intermediate scores [T,E]);
 * the benchmark tables name the softmax and sigmoid score functions.
 *
 * Per token row x (length E):
 *   score     softmax: s = exp(x - max x) / sum exp(x - max x)  (all E experts)
 *             sigmoid: s = 1 / (1 + exp(-x))
 *   key       k = s + expert_bias (bias optional, used for selection only)
 *   groups    if num_groups > 1: E splits into num_groups contiguous groups;
 *             a group scores the sum of its K/group_topk largest keys; only
 *             the group_topk best groups stay selectable
 *   select    the K largest keys among selectable experts (ties: lower index)
 *   probs     softmax: c * s on selected experts, 0 elsewhere (no renormalising)
 *             sigmoid and post-softmax: c * s / (sum of s over the selected),
 *             0 elsewhere
 *   scores    s (fp32), every expert
 * with c = scaling_factor.
 *
 * logits       [T,E] dtype, input
 * expert_bias  [E] float or NULL
 * probs        [T,E] dtype, output
 * routing_map  [T,E] uint8 0/1, output, exactly K ones per row
 * scores       [T,E] float, output (saved for router_topk_bwd)
 *
 * MR_ERR_INVALID: T < 0, E < 1, K < 1, K > E, T*E > INT_MAX, unknown dtype or
 *   score_func, a NULL tensor when T > 0 (logits, probs, routing_map, scores),
 *   num_groups < 0, and for num_groups > 1: E % num_groups != 0,
 *   group_topk outside [1, num_groups], K % group_topk != 0 or
 *   K / group_topk > E / num_groups (PR #3012, Hardening: topk in [1, E] and
 *   topk % group_topk == 0; num_tokens * num_experts <= INT_MAX).
 *   num_groups 0 or 1 means no grouping (group_topk is then ignored).
 * MR_ERR_UNSUPPORTED: E > MR_MAX_EXPERTS, K > MR_MAX_TOPK,
 *   num_groups > MR_MAX_GROUPS.
 */
MR_API int router_topk_fwd(const void* logits, mr_dtype dtype, int T, int E, int K,
                    mr_score_func score_func, int num_groups, int group_topk,
                    float scaling_factor, const float* expert_bias, void* probs,
                    uint8_t* routing_map, float* scores, mr_stream_t stream);

/*
 * router_topk_fwd_compact — the same router forward with compact outputs:
 * per token, the K selected experts and their probabilities as [T, K] rows,
 * written alongside or instead of the dense [T, E] tensors.
 *
 * Source: ROCm/aiter PR #5652, "[HIP] [Perf] Fold shared-expert gate GEMV
 * into topk_softmax kernel", review (topk_softmax writes [T, K] weights,
 * indices and token_expert_indices; the weights and indices are addressed
 * through a row stride so that a caller can pass column views of wider
 * buffers; token_expert_indices is [T, K]); NVIDIA TensorRT-LLM PR #14592,
 * "[TRTLLM-12214][perf] DeepGemmFusedMoE: fuse masked gather +
 * finalize-scale into one Triton kernel" (the expanded row of token t's k-th
 * choice is t + k * num_rows).
 *
 * Row t, position k (0 <= k < K) holds the expert of rank k in the selection
 * order (key s + bias descending, index ascending):
 *   topk_weights[t * ld_weights + k]  its probability (as in probs), fp32
 *   topk_indices[t * ld_indices + k]  its index, int32
 *   token_expert_indices[t * K + k]   k * T + t (int32), when not NULL
 * Columns K .. ld - 1 of the weights and indices are left untouched.
 * probs, routing_map and scores are as in router_topk_fwd, each written only
 * when its pointer is not NULL: the map and the scores identical, the
 * probabilities of the renormalising score functions (sigmoid, post-softmax)
 * equal up to the order in which the K selected scores are summed.
 *
 * Errors: as router_topk_fwd, with probs, routing_map and scores optional;
 * MR_ERR_INVALID also for ld_weights < K, ld_indices < K, or NULL
 * logits / topk_weights / topk_indices when T > 0.
 */
MR_API int router_topk_fwd_compact(const void* logits, mr_dtype dtype, int T, int E, int K,
                                   mr_score_func score_func, int num_groups, int group_topk,
                                   float scaling_factor, const float* expert_bias,
                                   float* topk_weights, int ld_weights, int32_t* topk_indices,
                                   int ld_indices, int32_t* token_expert_indices, void* probs,
                                   uint8_t* routing_map, float* scores, mr_stream_t stream);

/*
 * router_expert_maps — the (expert, token)-sorted maps of [T, K] expert
 * choices: the permutation that groups the T K (token, choice) rows by
 * expert for the expert computation, and its inverse.
 *
 * Source: microsoft/onnxruntime PR #33366, "[CUDA] Add fused decode routing,
 * single-pass finalize, and PDL overlap for NVFP4 QMoE", Description item 1
 * ((expert, token)-sorted expert maps) and review (both row maps, expert ids
 * and expert offsets); NVIDIA TensorRT-LLM PR #14592, "[TRTLLM-12214][perf]
 * DeepGemmFusedMoE: fuse masked gather + finalize-scale into one Triton
 * kernel" (permuted_row = unpermuted_to_permuted[t + k * num_rows]; the
 * expert of a permuted row and its column permuted_row -
 * expert_first_token_offset[expert]).
 *
 * The choice (t, k) is the expanded row u = t + k T.  Choices are ordered by
 * expert ascending, then token ascending; permuted row p is the p-th choice.
 *   expert_first_token_offset [E+1] int32: first permuted row of expert e;
 *                             entry E is the number of choices placed
 *   permuted_to_unpermuted    [T K] int32: the expanded row u of row p
 *   unpermuted_to_permuted    [T K] int32: the permuted row of u
 *   permuted_experts          [T K] int32: the expert of row p
 * topk_indices [T, ld_indices] int32 (the first K columns are read), e.g.
 * from router_topk_fwd_compact.  Each row should name K distinct experts: a
 * repeated expert leaves the maps unspecified (never written out of range).
 * An index outside [0, E) is skipped: its unpermuted_to_permuted entry is -1
 * and it takes no permuted row.
 * workspace: device memory of router_expert_maps_workspace_bytes(T, E)
 * bytes, 16-byte aligned; its contents need no initialisation.  On the
 * stream: a one-block kernel that zeroes a counter and one cooperative
 * launch when the batch's 64-token tiles fit on the GPU at once, else three
 * launches; deterministic either way (identical results).
 *
 * MR_ERR_INVALID: T < 0, E < 1, K < 1, K > E, ld_indices < K, T*E > INT_MAX,
 *   a NULL pointer when T > 0, a small or misaligned workspace.
 * MR_ERR_UNSUPPORTED: E > MR_MAX_EXPERTS or K > MR_MAX_TOPK.
 * T = 0: nothing is written.
 */
MR_API size_t router_expert_maps_workspace_bytes(int T, int E);
MR_API int router_expert_maps(const int32_t* topk_indices, int ld_indices, int T, int E, int K,
                              int32_t* expert_first_token_offset,
                              int32_t* permuted_to_unpermuted, int32_t* unpermuted_to_permuted,
                              int32_t* permuted_experts, void* workspace, size_t workspace_bytes,
                              mr_stream_t stream);

/*
 * router_topk_fwd_maps — router_topk_fwd_compact followed by
 * router_expert_maps of its indices.  Up to 8 tokens (decode) with 16-byte
 * aligned logits (and bias) and E % 4 == 0 (fp32) or E % 8 == 0 (bf16), it is
 * one kernel launch in one block: the rows are routed by the block's warps
 * and the block then builds the maps, as the fused decode routing of
 * onnxruntime PR #33366 (Description item 1) does; the workspace is then not
 * used and may be NULL.  Otherwise it is the compact forward plus the three
 * map launches, with the workspace of router_expert_maps.
 *
 * Arguments and outputs: those of router_topk_fwd_compact (no dense
 * outputs) and router_expert_maps; errors as both.
 */
MR_API int router_topk_fwd_maps(const void* logits, mr_dtype dtype, int T, int E, int K,
                                mr_score_func score_func, int num_groups, int group_topk,
                                float scaling_factor, const float* expert_bias,
                                float* topk_weights, int ld_weights, int32_t* topk_indices,
                                int ld_indices, int32_t* token_expert_indices,
                                int32_t* expert_first_token_offset,
                                int32_t* permuted_to_unpermuted,
                                int32_t* unpermuted_to_permuted, int32_t* permuted_experts,
                                void* workspace, size_t workspace_bytes, mr_stream_t stream);

/*
 * router_topk_bwd — gradient of the forward's probs with respect to logits.
 *
 * Source: TransformerEngine PR #3012, Backward kernels (pass 1: per-row sums
 * by register and warp reduction; pass 2: per-element gradients) and the
 * review summary (the gradient per score function).  The selection and the
 * expert bias carry no gradient.  With g = grad_probs, m = routing_map,
 * s = scores and c = scaling_factor, per row:
 *   softmax: D = c * sum_j m_j g_j s_j;   gx_j = s_j * (c m_j g_j - D)
 *   sigmoid: S = sum_j m_j s_j, D = sum_j m_j g_j s_j;
 *            gx_j = m_j * (c / S) * (g_j - D / S) * s_j * (1 - s_j)
 *   post-softmax (s the full softmax): S, D as for sigmoid;
 *            gx_j = m_j * (c / S) * (g_j - D / S) * s_j
 *
 * grad_probs   [T,E] dtype, input
 * routing_map  [T,E] uint8 (nonzero = selected), input from router_topk_fwd
 * scores       [T,E] float, input from router_topk_fwd
 * grad_logits  [T,E] dtype, output
 * K            the forward's K (checked, 1 <= K <= E)
 *
 * MR_ERR_INVALID / MR_ERR_UNSUPPORTED: as router_topk_fwd for T, E, K, dtype,
 *   score_func and NULL tensors.  A sigmoid row whose map selects nothing
 *   produces NaN (S = 0); the forward never writes such a map.
 */
MR_API int router_topk_bwd(const void* grad_probs, const uint8_t* routing_map,
                    const float* scores, mr_dtype dtype, int T, int E, int K,
                    mr_score_func score_func, float scaling_factor,
                    void* grad_logits, mr_stream_t stream);

/*
 * router_aux_scores_fwd — full-row scores for the load-balancing aux loss,
 * with their top-K routing map.
 *
 * Source: TransformerEngine PR #3012, Summary (fused_score_for_moe_aux_loss)
 * and the aux_loss rows of both benchmark tables.  Per row:
 *   softmax: q = softmax(x)
 *   sigmoid: sig = 1 / (1 + exp(-x)),  q = sig / sum_E sig
 *   routing_map = top-K of q (ties: lower index; no bias, groups or scaling)
 *
 * logits        [T,E] dtype, input
 * scores        [T,E] float, output q
 * routing_map   [T,E] uint8 0/1, output
 * intermediate  [T,E] float, output sig (sigmoid: required; softmax: may be
 *               NULL, and if given receives q again)
 *
 * Errors: as router_topk_fwd for T, E, K, dtype, score_func (MR_SOFTMAX_POST
 *   is MR_ERR_INVALID here); when T > 0, NULL
 *   logits, scores or routing_map, or NULL intermediate with sigmoid:
 *   MR_ERR_INVALID.
 */
MR_API int router_aux_scores_fwd(const void* logits, mr_dtype dtype, int T, int E,
                          int K, mr_score_func score_func, float* scores,
                          uint8_t* routing_map, float* intermediate,
                          mr_stream_t stream);

/*
 * router_aux_scores_bwd — gradient of the aux scores q with respect to logits.
 *
 * Source: TransformerEngine PR #3012, Summary and Backward kernels (same
 * two-pass structure as the top-K backward).  With g = grad_scores, per row:
 *   softmax (saved = q):   gx_j = q_j * (g_j - sum_i g_i q_i)
 *   sigmoid (saved = sig): Z = sum_i sig_i, Dq = sum_i g_i sig_i / Z,
 *                          gx_j = (g_j - Dq) / Z * sig_j * (1 - sig_j)
 *
 * grad_scores  [T,E] float, input
 * saved        [T,E] float: softmax the forward's scores, sigmoid its
 *              intermediate
 * grad_logits  [T,E] dtype, output
 * K            the forward's K (checked, 1 <= K <= E; not otherwise used)
 *
 * Errors: as router_topk_bwd.
 */
MR_API int router_aux_scores_bwd(const float* grad_scores, const float* saved,
                          mr_dtype dtype, int T, int E, int K,
                          mr_score_func score_func, void* grad_logits,
                          mr_stream_t stream);

/*
 * router_aux_loss_fwd — the load-balancing aux loss over the aux-score
 * forward's outputs, with the tokens routed to each expert.
 *
 * Source: TransformerEngine PR #3012, Important Files Changed
 * (fused_moe_aux_loss: the page names the op; its formula is not printed).
 * The loss taken here is the standard load-balancing loss
 *   loss = coeff * E * sum_e f_e * P_e,  f_e = tokens_e / (T K),
 *   P_e = (1/T) sum_t q_te,  tokens_e = sum_t map_te,
 * i.e. coeff * E / (K T^2) * sum_e (sum_t q_te) * tokens_e.
 *
 * aux_scores         [T,E] float q (router_aux_scores_fwd's scores), input
 * routing_map        [T,E] uint8, nonzero = routed, input
 * loss               [1] float, output (device memory)
 * tokens_per_expert  [E] int32, output
 * workspace          device scratch of at least
 *                    router_aux_loss_workspace_bytes(T, E) bytes, 16-byte
 *                    aligned, owned by the caller; its contents need no
 *                    initialisation and are overwritten
 *
 * A one-block kernel that zeroes the workspace's counters, then one kernel,
 * both on `stream`; the reduction order is fixed (compensated fp32 sums, no
 * floating-point atomics) and depends on T, E and the row layout only, so
 * repeated calls give identical bits.  T == 0 is a no-op (nothing written).
 * MR_ERR_INVALID: T < 0, E < 1, K outside [1, E], T*E > INT_MAX, a NULL
 * pointer when T > 0, a workspace too small or misaligned.
 * MR_ERR_UNSUPPORTED: E > MR_MAX_EXPERTS.
 */
MR_API size_t router_aux_loss_workspace_bytes(int T, int E);
MR_API int router_aux_loss_fwd(const float* aux_scores, const uint8_t* routing_map, int T, int E,
                               int K, float coeff, float* loss, int32_t* tokens_per_expert,
                               void* workspace, size_t workspace_bytes, mr_stream_t stream);

/*
 * router_aux_loss_bwd — gradient of the aux loss with respect to the aux
 * scores: grad_aux_scores[t, e] = grad_loss * coeff E / (K T^2) * tokens_e
 * (the loss is linear in q; the token counts carry no gradient).
 *
 * grad_loss          [1] float, device memory, input
 * tokens_per_expert  [E] int32 from router_aux_loss_fwd, input
 * grad_aux_scores    [T,E] float, output
 * Errors: as router_aux_loss_fwd (no workspace).
 */
MR_API int router_aux_loss_bwd(const float* grad_loss, const int32_t* tokens_per_expert, int T,
                               int E, int K, float coeff, float* grad_aux_scores,
                               mr_stream_t stream);

/*
 * router_aux_loss_fwd_noalloc — router_aux_loss_fwd without a workspace.
 * The paper has no counterpart: this entry point exists for callers that
 * cannot allocate device memory at the point of the call.  Examples: a
 * runtime whose memory plan reserves all device memory up front, so that a
 * cudaMalloc fails or bypasses its accounting; a plain C caller with no
 * allocator to hand a workspace from; code that must not pay the implicit
 * device synchronisation of cudaFree after the call.
 *
 * The column partials go to a fixed device array inside this library of
 * MR_AUX_LOSS_NOALLOC_SCRATCH_BYTES (1,180,688 bytes: up to
 * MR_AUX_LOSS_NOALLOC_BLOCKS partial rows for E up to MR_MAX_EXPERTS, and a
 * small tail for the reduction's last step).  Every
 * GPU that loads the library holds that array until the process exits.  The
 * call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.  The caller still owns and passes every input and output.
 *
 * Arguments, layouts, results and errors are those of router_aux_loss_fwd
 * without workspace/workspace_bytes; E beyond what the array holds returns
 * MR_ERR_UNSUPPORTED.  The loss and tokens equal router_aux_loss_fwd's bit
 * for bit (the same kernel, partial rows and summation order); repeated
 * calls on the same inputs give the same bits.
 *
 * Set-up: the first call on a device (that device current) looks up the
 * array's device address, once per device; make that first call before any
 * stream capture begins.  Sharing: every call on a device uses the same
 * array, which keeps the last call's contents (nothing needs clearing: each
 * call writes every partial it reads before reading it and zeroes its own
 * completion counters).  Calls whose work
 * overlaps on the GPU — on two streams, or from two host threads — race on
 * the array and give wrong results; order them on one stream or with
 * events.
 */
#define MR_AUX_LOSS_NOALLOC_BLOCKS 64
#define MR_AUX_LOSS_NOALLOC_SCRATCH_BYTES \
  ((size_t)MR_AUX_LOSS_NOALLOC_BLOCKS * MR_MAX_EXPERTS * 8u + 1040u)
MR_API int router_aux_loss_fwd_noalloc(const float* aux_scores, const uint8_t* routing_map, int T,
                                       int E, int K, float coeff, float* loss,
                                       int32_t* tokens_per_expert, mr_stream_t stream);

/* Static English text for a status code (never NULL). */
MR_API const char* moe_router_strerror(int code);

/*
 * Kernel path of the top-K and aux forwards.
 *   MR_PATH_SEGMENT: the row of logits lives in the registers of 8, 16 or 32
 *     lanes of a warp (every shape, bias and groups included);
 *   MR_PATH_STAGED: each warp streams rows through shared memory with bulk
 *     copies (bias and groups included; E % 4 == 0 for fp32, E % 8 == 0 for
 *     bf16; 16-byte aligned tensors).  router_topk_fwd_maps's one-launch
 *     decode form always runs on this path;
 *   MR_PATH_REGISTER: rows arrive by bulk copy like the staged path and are
 *     then held in the registers of one warp, the K-th largest key found
 *     by bisection over compacted candidates (router_topk_fwd,
 *     router_topk_fwd_compact and router_aux_scores_fwd with E <= 512, the
 *     staged path's alignment; bias allowed, groups when each is a
 *     power-of-two number of 4-expert chunks and sums at most 4 keys).
 * MR_PATH_AUTO takes the register path where it applies (for compact
 * outputs only with bias or groups) and the staged path elsewhere, except
 * for batches of 8192 or more tokens with E < 128 (the segment path is
 * faster there).  A forced path that does not apply to a
 * call falls back to the automatic choice.  Process-wide; meant for tests and
 * benchmarks.  The environment variable MOE_ROUTER_FORCE_PATH
 * (auto|segment|staged|register) sets the initial value.  Returns the
 * previous value, or MR_ERR_INVALID for an unknown path.
 */
typedef enum {
  MR_PATH_AUTO = 0,
  MR_PATH_SEGMENT = 1,
  MR_PATH_STAGED = 2,
  MR_PATH_REGISTER = 3
} mr_path;
MR_API int moe_router_force_path(int path);

/*
 * Lanes that share one token row in the segment forward: 8, 16 or 32, or 0
 * for the automatic choice (the default).  A width that cannot hold a given
 * row (too few lanes for its E, or 2 * lanes < K) falls back to the
 * automatic choice for that call.  Process-wide; meant for tests and
 * benchmarks.  Returns the previous value, or MR_ERR_INVALID.
 */
MR_API int moe_router_force_fwd_lanes(int lanes);

/*
 * Device status of the current device: 0, or 1 when a kernel gave up a
 * bounded wait for a bulk copy (about one second) and returned early, leaving
 * its outputs incomplete.  Reading clears the word.  Synchronous: it waits
 * for the device's outstanding work (a blocking cudaMemcpy).
 */
MR_API int moe_router_device_status(int* status);

/*
 * Diagnostic for the failure path above: enqueue one small kernel that waits,
 * with the same bounded wait the router kernels use, for a barrier phase that
 * nothing completes.  After about timeout_us microseconds (1..1000000) the
 * wait gives up and the device status word becomes 1, which
 * moe_router_device_status then reports (and clears).  No fault, trap or hang
 * is involved: the kernel simply returns.  MR_ERR_INVALID for timeout_us out
 * of range.
 */
MR_API int moe_router_selftest_bounded_wait(unsigned timeout_us, mr_stream_t stream);

/* Library ABI version: 100 * major + minor. */
MR_API int moe_router_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTER_H */
