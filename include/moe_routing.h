/*
 * moe_routing.h -- C ABI of libmoe_routing.so, the GB300 (sm_103a) MoE
 * routing and combine hot path: group-limited top-k router, expert index
 * builder, and fused unpermute + weighted top-k sum.
 *
 * Sources (Mojo kernel library API pages, cited by page title and section):
 *   "group_limited_router_kernel"  -> moe_route
 *   "moe_create_indices"           -> moe_create_indices (fused with the
 *                                     router: moe_route_index)
 *   "moe_finalize"                 -> moe_finalize
 *
 * Conventions for every entry point:
 *   - Argument order follows the pages: outputs first, then inputs, then the
 *     sizes that the pages carry as tensor shapes or compile-time parameters,
 *     then the CUDA stream that replaces the pages' DeviceContext.
 *   - Every pointer is a DEVICE pointer to a dense row-major buffer owned by
 *     the caller. The library allocates nothing, frees nothing and keeps no
 *     state between calls; the index builder's scratch space is a
 *     caller-provided workspace (moe_route_index keeps counts there that every
 *     call leaves at zero, moe_route_index_single_launch a call counter).
 *   - Every call only enqueues work on `stream` (0 = the legacy default
 *     stream) and returns without synchronising, except
 *     moe_read_device_status, which waits for the stream.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and reported as a moe_status_t. MOE_ERR_CUDA means a launch failed
 *     (cudaGetLastError after the launch). Errors found in the DATA (an
 *     expert id outside [0, n_experts), a restore_order entry outside
 *     [0, T*K)) are recorded in a device status word and never trap; see
 *     moe_read_device_status.
 *   - A call with zero tokens / slots is valid.
 */
#ifndef MOE_ROUTING_H
#define MOE_ROUTING_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

/* Raw bf16 bit pattern (1 sign, 8 exponent, 7 mantissa bits), as in __nv_bfloat16. */
typedef uint16_t moe_bf16_t;

/* Element types of the dtype-generic entry points. */
typedef enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 } moe_dtype_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULL_PTR = 1,     /* a required pointer is NULL */
  MOE_ERR_INVALID_ARG = 2,  /* sizes inconsistent with the method (e.g. E % n_groups != 0) */
  MOE_ERR_MISALIGNED = 3,   /* a pointer breaks the stated alignment */
  MOE_ERR_UNSUPPORTED = 4,  /* valid for the method but outside this library's limits */
  MOE_ERR_CUDA = 5,         /* a CUDA launch or copy failed */
  MOE_ERR_WORKSPACE = 6,    /* workspace NULL or smaller than the size query returns */
  MOE_ERR_DEVICE_DATA = 7   /* moe_read_device_status: the device status word is not 0 */
} moe_status_t;

/* Bits of the device status word written by moe_create_indices, moe_route_index
 * and (when given a status pointer) moe_finalize_ex and moe_permute. */
#define MOE_DEVICE_STATUS_BAD_EXPERT_ID 0x1u /* some topk_ids entry was outside [0, E) */
#define MOE_DEVICE_STATUS_SYNC_TIMEOUT 0x2u  /* single-launch route+index: a cross-CTA wait gave up */
#define MOE_DEVICE_STATUS_SYNC_STATE 0x4u    /* route+index: inconsistent counts (workspace not zero-filled) */
#define MOE_DEVICE_STATUS_BAD_RESTORE_ORDER 0x8u /* finalize/permute: an entry >= T*K */

/* Limits of this implementation. */
#define MOE_MAX_EXPERTS 1024       /* n_routed_experts / n_experts */
#define MOE_MAX_GROUPS 32          /* n_groups */
#define MOE_MAX_EXPERTS_PER_TOK 32 /* n_experts_per_tok / num_experts_per_token */
/* Row granularity of the per-expert scale blocks reported through scales_offset_p. */
#define MOE_SCALES_ROW_ALIGNMENT 128

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status_t status);

/*
 * moe_route -- group-limited top-k router.
 * Page "group_limited_router_kernel": description paragraph; Parameters
 * n_routed_experts, n_experts_per_tok, n_groups, topk_group, norm_weights;
 * Args expert_indices, expert_weights, expert_scores, expert_bias,
 * routed_scaling_factor.
 *
 * For each token t (row of expert_scores):
 *   b[e]  = expert_scores[t,e] + expert_bias[e]           (fp32, selection only)
 *   g[j]  = largest + second-largest b[e] of group j       (group j = experts
 *           j*S .. j*S+S-1, S = E / n_groups; g[j] = b if S == 1)
 *   keep the topk_group groups with the largest g (ties -> lower group index)
 *   expert_indices[t,:] = the n_experts_per_tok experts of the kept groups
 *           with the largest b, in that order (ties -> lower expert index)
 *   expert_weights[t,k] = expert_scores[t, expert_indices[t,k]]; if
 *           norm_weights, divided by their fp32 sum taken in k order; then
 *           multiplied by routed_scaling_factor. All fp32, round-to-nearest.
 *
 * expert_indices  [T, K] int32 out.   expert_weights [T, K] fp32 out.
 * expert_scores   [T, E] fp32 in.     expert_bias    [E] fp32 in.
 * Requirements: 1 <= E <= MOE_MAX_EXPERTS; 1 <= n_groups <= MOE_MAX_GROUPS and
 * E % n_groups == 0; 1 <= topk_group <= n_groups; 1 <= K <= topk_group * S and
 * K <= MOE_MAX_EXPERTS_PER_TOK; T >= 0. 4-byte aligned pointers (16-byte
 * alignment of expert_scores with E % 4 == 0 enables vector loads). Scores and
 * bias must be free of NaN (the selection is then unspecified, never faulting).
 */
moe_status_t moe_route(int32_t* expert_indices, float* expert_weights,
                       const float* expert_scores, const float* expert_bias,
                       int64_t num_tokens, int32_t n_routed_experts, int32_t n_experts_per_tok,
                       int32_t n_groups, int32_t topk_group, int32_t norm_weights,
                       float routed_scaling_factor, cudaStream_t stream);

/* Score loaders of moe_route_ex (the page's scores_input_fn). */
typedef enum {
  MOE_SCORES_AS_GIVEN = 0, /* the score is the loaded value (moe_route) */
  MOE_SCORES_SIGMOID = 1,  /* the score is sigmoid(loaded logit) */
  MOE_SCORES_SOFTMAX = 2   /* the scores are the softmax of the token's logits */
} moe_score_fn_t;

/*
 * moe_route_ex -- moe_route with a fused score loader.
 * Page "group_limited_router_kernel": Parameters scores_input_fn (an optional
 * loader of the score of a (token, expert) pair; without it scores load from
 * expert_scores).
 *
 * With MOE_SCORES_SIGMOID, expert_scores holds gate logits x and every score
 * (for selection and for the weights) is sigmoid(x) = 1 / (1 + exp(-x)) in
 * fp32, computed as the load happens, so the activated [T, E] tensor is never
 * written. exp is the library's own: x clamped to [-87, 88], Cody-Waite
 * reduction by ln2 (head 0.693145751953125, tail 1.42860682030941723e-6),
 * degree-7 Taylor polynomial in Horner form with fused multiply-adds, times
 * 2^n; within a few ulp of the true value, and reproducible bit for bit.
 * With MOE_SCORES_SOFTMAX, the scores of a token are the softmax of its E
 * logits, exp(x - max) / sum, with that exp, fp32 throughout, and the sum taken
 * in ascending expert order (the plainest reading: the page gives no order),
 * so the result is reproducible bit for bit as well.
 * Everything else is as in moe_route. An unknown score_fn returns
 * MOE_ERR_UNSUPPORTED.
 */
moe_status_t moe_route_ex(int32_t* expert_indices, float* expert_weights,
                          const float* expert_scores, const float* expert_bias,
                          int64_t num_tokens, int32_t n_routed_experts, int32_t n_experts_per_tok,
                          int32_t n_groups, int32_t topk_group, int32_t norm_weights,
                          float routed_scaling_factor, moe_score_fn_t score_fn,
                          cudaStream_t stream);

/*
 * Workspace bytes that moe_create_indices needs for num_slots slots and
 * n_experts experts (always >= 256). Host-only; never fails (returns 0 for
 * negative num_slots or n_experts outside [1, MOE_MAX_EXPERTS]).
 */
size_t moe_create_indices_workspace_size(int64_t num_slots, int32_t n_experts);

/*
 * moe_create_indices -- bucket sort of the flat router output by expert.
 * Page "moe_create_indices": description paragraph (bucket sort so that each
 * expert's tokens are contiguous); Parameters expected_count (no per-expert
 * limit here); Args token_expert_order, expert_start_indices,
 * restore_token_order, expert_ids, expert_usage_stats, topk_ids,
 * scales_offset_p.
 *
 * Slot i = t*K + k of the flattened topk_ids [T, K] (num_slots = T*K):
 *   token_expert_order [N]  uint32 out: slot indices grouped by expert, experts
 *        in ascending id, ascending slot index within one expert (stable).
 *   restore_token_order [N] uint32 out: position of slot i in
 *        token_expert_order (its inverse permutation).
 *   expert_ids [E] int32 out: the A active experts (count > 0) in ascending
 *        id, then -1 in entries A .. E-1.
 *   expert_start_indices [E+1] uint32 out: compact CSR over expert_ids: entry j
 *        < A is where expert_ids[j]'s slots start, entries A .. E are N.
 *   expert_usage_stats [2] uint32 out: {max slots on one expert, A}.
 *   topk_ids [N] int32 in: expert id of each slot.
 * workspace: device buffer of at least moe_create_indices_workspace_size()
 *   bytes, 256-byte aligned, caller-owned; its first 4 bytes receive the
 *   device status word. Calls sharing one workspace must not overlap.
 * scales_offset_p (optional, may be NULL) [E+1] uint32 out: the aligned scale
 *   offsets for an FP8/block-scaled grouped matmul. The page does not give the
 *   alignment; here every active expert's rows are padded to a multiple of
 *   MOE_SCALES_ROW_ALIGNMENT, the row granularity of block-scaled tensor-core
 *   scale-factor layouts: entry j < A = sum over active experts j' < j of
 *   ceil(count_j' / 128) * 128, entries A .. E = that padded total. Requires
 *   N + 127 * E < 2^32 (else MOE_ERR_UNSUPPORTED).
 * Requirements: 0 <= N < 2^32 - 1; 1 <= E <= MOE_MAX_EXPERTS; 4-byte aligned
 * buffers. Out-of-range ids set MOE_DEVICE_STATUS_BAD_EXPERT_ID, are left out
 * of every output count and leave the contents of the outputs unspecified.
 */
moe_status_t moe_create_indices(uint32_t* token_expert_order, uint32_t* expert_start_indices,
                                uint32_t* restore_token_order, int32_t* expert_ids,
                                uint32_t* expert_usage_stats, const int32_t* topk_ids,
                                int64_t num_slots, int32_t n_experts, void* workspace,
                                size_t workspace_bytes, uint32_t* scales_offset_p,
                                cudaStream_t stream);

/*
 * Workspace bytes that moe_route_index needs for num_tokens tokens,
 * n_routed_experts experts and n_experts_per_tok experts per token (always
 * >= 4864). Host-only; returns 0 for negative num_tokens, n_routed_experts
 * outside [1, MOE_MAX_EXPERTS] or n_experts_per_tok outside
 * [1, MOE_MAX_EXPERTS_PER_TOK].
 */
size_t moe_route_index_workspace_size(int64_t num_tokens, int32_t n_routed_experts,
                                      int32_t n_experts_per_tok);

/*
 * moe_route_index -- moe_route_ex followed by moe_create_indices on its
 * output, with the router counting its own output.
 * Pages "group_limited_router_kernel" (the routing: as moe_route and
 * moe_route_ex) and "moe_create_indices" (the index: as moe_create_indices
 * with topk_ids = expert_indices and num_slots = T*K). The pages launch the
 * two as separate kernels; fusing the count into the router is this
 * library's design.
 *
 * Every output is bit-identical to those of the two separate calls:
 * expert_indices [T, K] int32 and expert_weights [T, K] fp32 (written, and
 * also read back by the index build); token_expert_order [T*K],
 * restore_token_order [T*K], expert_start_indices [E+1], expert_ids [E],
 * expert_usage_stats [2] and the optional scales_offset_p [E+1] as described
 * at moe_create_indices. Arguments and requirements are the union of
 * moe_route_ex's and moe_create_indices', plus T*K < 2^32 - 1.
 *
 * Execution: the router adds each of its slots to a count per (expert,
 * 1024-slot chunk) with a relaxed atomic (integer sums do not depend on the
 * order, so the result is deterministic); a row-prefix kernel and the scatter
 * kernel of moe_create_indices follow. Three launches in all (two when
 * T*K <= 1024), no waits between CTAs.
 * workspace: device buffer of at least moe_route_index_workspace_size()
 *   bytes, 256-byte aligned, caller-owned, ZERO-FILLED before its first use
 *   (e.g. cudaMemset): the router's counts accumulate into it, and every call
 *   leaves them zero again, so the workspace is zeroed once, not per call.
 *   Counts that do not add up to T*K (a workspace that was not zero-filled)
 *   set MOE_DEVICE_STATUS_SYNC_STATE; the index outputs are then unspecified,
 *   no position at or past T*K is written, and the call leaves the counts it
 *   used zero, so the next call on the same shapes is correct again.
 *   The prefix matrix is placed at the end of workspace_bytes, so one
 *   workspace may serve calls of any shapes that fit it, in any order.
 *   Word 0 receives the device status word (moe_read_device_status). Calls
 *   sharing one workspace must not overlap, and a workspace serves
 *   moe_route_index or moe_route_index_single_launch, not both.
 */
moe_status_t moe_route_index(int32_t* expert_indices, float* expert_weights,
                             uint32_t* token_expert_order, uint32_t* expert_start_indices,
                             uint32_t* restore_token_order, int32_t* expert_ids,
                             uint32_t* expert_usage_stats, const float* expert_scores,
                             const float* expert_bias, int64_t num_tokens,
                             int32_t n_routed_experts, int32_t n_experts_per_tok,
                             int32_t n_groups, int32_t topk_group, int32_t norm_weights,
                             float routed_scaling_factor, moe_score_fn_t score_fn,
                             void* workspace, size_t workspace_bytes, uint32_t* scales_offset_p,
                             cudaStream_t stream);

/*
 * Workspace bytes that moe_route_index_single_launch needs (always >= 2048).
 * Host-only; returns 0 for negative num_tokens or n_routed_experts outside
 * [1, MOE_MAX_EXPERTS].
 */
size_t moe_route_index_single_launch_workspace_size(int64_t num_tokens,
                                                    int32_t n_routed_experts);

/*
 * moe_route_index_single_launch -- the same outputs as moe_route_index from
 * ONE cooperative kernel launch. On the measured shapes it is the slower of
 * the two (DeepSeek-V3-shaped prefill, 16384 tokens: 31.6 us against 19.5 us
 * for moe_route_index on one GB300); it suits callers that want a single
 * launch per batch.
 * Every output is bit-identical to those of the two separate calls:
 * expert_indices [T, K] int32 and expert_weights [T, K] fp32 (written, and
 * also read back by the index build); token_expert_order [T*K],
 * restore_token_order [T*K], expert_start_indices [E+1], expert_ids [E],
 * expert_usage_stats [2] and the optional scales_offset_p [E+1] as described
 * at moe_create_indices. Arguments and requirements are the union of
 * moe_route_ex's and moe_create_indices', plus T*K < 2^32 - 1.
 *
 * workspace: device buffer of at least
 *   moe_route_index_single_launch_workspace_size() bytes, 256-byte aligned,
 *   caller-owned, ZERO-FILLED before its first use (e.g. cudaMemset). Word 0
 *   receives the device status word (read it with moe_read_device_status);
 *   word 1 counts the calls made on the workspace;
 *   the next 1024 bytes hold progress counters that each call zeroes for
 *   the next one.
 *   The CTAs of a call exchange their counts through words tagged with that
 *   call's number, so nothing needs clearing between calls. Calls sharing one
 *   workspace must not overlap. The call number is 32 bits wide (after
 *   0xFFFFFFFF it continues at 2): zero-fill the workspace again at least
 *   once every 2^31 calls, so that no word left by a call 2^32 calls earlier
 *   can carry a current number.
 * Execution: one cooperative launch (all CTAs resident at once; CTAs of up
 *   to 1024 threads, at most one per 8 tokens). Every cross-CTA wait gives up
 *   after one second; the call then sets MOE_DEVICE_STATUS_SYNC_TIMEOUT and
 *   leaves the index outputs unspecified. MOE_DEVICE_STATUS_SYNC_STATE means
 *   the exchanged counts were inconsistent, which only a workspace that was
 *   not zero-filled can cause. After either bit, zero-fill the workspace
 *   before the next call.
 * Returns MOE_ERR_UNSUPPORTED when the kernel cannot be made resident (no
 *   CTA fits on an SM), and MOE_ERR_CUDA when the cooperative launch fails.
 */
moe_status_t moe_route_index_single_launch(
    int32_t* expert_indices, float* expert_weights, uint32_t* token_expert_order,
    uint32_t* expert_start_indices, uint32_t* restore_token_order, int32_t* expert_ids,
    uint32_t* expert_usage_stats, const float* expert_scores, const float* expert_bias,
    int64_t num_tokens, int32_t n_routed_experts, int32_t n_experts_per_tok, int32_t n_groups,
    int32_t topk_group, int32_t norm_weights, float routed_scaling_factor,
    moe_score_fn_t score_fn, void* workspace, size_t workspace_bytes, uint32_t* scales_offset_p,
    cudaStream_t stream);

/*
 * moe_finalize -- fused unpermute gather + top-k weighted row sum.
 * Page "moe_finalize": description paragraph (gather each token's K rows of
 * down through restore_order, scale by the router weight, accumulate in
 * fp32, never materialise [T, K, H]); Args output, down, restore_order,
 * router_weight.
 *
 *   output[t,h] = bf16_rn( sum_{k=0}^{K-1} router_weight[t,k] *
 *                          float(down[restore_order[t*K+k], h]) )
 * accumulated in fp32 in k order with fused multiply-add from 0.
 *
 * output [T, H] bf16 out. down [T*K, H] bf16 in, rows in token_expert_order
 * order. restore_order [T*K] uint32 in. router_weight [T, K] fp32 in.
 * Requirements: T >= 0; 1 <= K <= MOE_MAX_EXPERTS_PER_TOK; T*K < 2^32; H >= 0
 * and H % 8 == 0; output and down 16-byte aligned; restore_order and
 * router_weight 4-byte aligned; output must not overlap down. A
 * restore_order entry >= T*K is skipped (contributes nothing) and never read;
 * moe_finalize_ex can also report it.
 */
moe_status_t moe_finalize(moe_bf16_t* output, const moe_bf16_t* down,
                          const uint32_t* restore_order, const float* router_weight,
                          int64_t num_tokens, int32_t num_experts_per_token, int64_t hidden,
                          cudaStream_t stream);

/*
 * moe_finalize_ex -- moe_finalize with the router-weight and output element
 * types as arguments.
 * Page "moe_finalize": Parameters weight_type and out_type (the page's
 * kernel is generic over them; down_type stays bf16 here).
 *
 * Same sum as moe_finalize, accumulated in fp32 (a bf16 weight widens to fp32
 * exactly). output_dtype MOE_DTYPE_BF16 rounds each sum to nearest-even bf16;
 * MOE_DTYPE_F32 stores the fp32 sum itself.
 * output [T, H] of output_dtype, 16-byte aligned. router_weight [T, K] of
 * weight_dtype, aligned to its element size. Other arguments and rules as in
 * moe_finalize; an unknown dtype returns MOE_ERR_UNSUPPORTED.
 * device_status: optional device pointer (4-byte aligned, or NULL). When
 *   given, a restore_order entry >= T*K, which is skipped as in moe_finalize,
 *   also ORs MOE_DEVICE_STATUS_BAD_RESTORE_ORDER into *device_status (never a
 *   fault or a trap). The word is not cleared by the call: zero it first, and
 *   read it with moe_read_device_status.
 */
moe_status_t moe_finalize_ex(void* output, moe_dtype_t output_dtype, const moe_bf16_t* down,
                             const uint32_t* restore_order, const void* router_weight,
                             moe_dtype_t weight_dtype, int64_t num_tokens,
                             int32_t num_experts_per_token, int64_t hidden,
                             uint32_t* device_status, cudaStream_t stream);

/*
 * moe_permute -- expert-contiguous copy of the token rows, the input of the
 * grouped matmul that sits between moe_create_indices and moe_finalize.
 * Page "moe_create_indices": description paragraph (tokens are grouped by
 * expert so that downstream kernels such as grouped matmul can process each
 * expert's tokens contiguously).
 *
 *   permuted[restore_token_order[t*K+k], :] = input[t, :]   for t < T, k < K
 * so row p of permuted is input[token_expert_order[p] / K].
 *
 * permuted [T*K, H] bf16 out. input [T, H] bf16 in. restore_token_order
 * [T*K] uint32 in (as written by moe_create_indices).
 * Requirements: T >= 0; 1 <= K <= MOE_MAX_EXPERTS_PER_TOK; T*K < 2^32; H >= 0
 * and H % 8 == 0; permuted and input 16-byte aligned and not overlapping;
 * restore_token_order 4-byte aligned. An entry >= T*K is skipped; with a
 * device_status pointer (optional, 4-byte aligned, or NULL) it also ORs
 * MOE_DEVICE_STATUS_BAD_RESTORE_ORDER into *device_status, as moe_finalize_ex.
 */
moe_status_t moe_permute(moe_bf16_t* permuted, const moe_bf16_t* input,
                         const uint32_t* restore_token_order, int64_t num_tokens,
                         int32_t num_experts_per_token, int64_t hidden, uint32_t* device_status,
                         cudaStream_t stream);

/*
 * Reads a device status word: word 0 of the workspace that the last
 * moe_create_indices or moe_route_index call on it wrote, or a status word
 * given to moe_create_indices_no_alloc, moe_finalize_ex or moe_permute
 * (0 = clean; MOE_DEVICE_STATUS_* bits otherwise). Enqueues a 4-byte copy on
 * `stream` and waits for the stream to finish. Writes the word to
 * *host_status and returns MOE_OK when it is 0, MOE_ERR_DEVICE_DATA when it
 * is not.
 */
moe_status_t moe_read_device_status(const void* workspace, uint32_t* host_status,
                                    cudaStream_t stream);

/*
 * moe_create_indices_no_alloc -- the same index build as moe_create_indices,
 * for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point.
 *
 * Why: some callers can hand a kernel only the tensors it declares as inputs
 * and outputs. One example is an operator inside a framework whose memory
 * pool owns all device memory and offers no scratch request. Another is a
 * serving loop that reserves memory at start-up and must not call cudaMalloc
 * on the request path. Such callers cannot provide moe_create_indices'
 * workspace. This variant keeps its scratch in a file-scope __device__
 * array of MOE_NO_ALLOC_SCRATCH_BYTES bytes inside the library. Every GPU
 * that loads the library holds that array until the process exits.
 *
 * Outputs, inputs and their requirements are those of moe_create_indices.
 * device_status: optional device pointer (4-byte aligned, or NULL) that
 *   receives the device status word (MOE_DEVICE_STATUS_* bits, 0 = clean).
 *   When it is NULL the word is written inside the scratch and cannot be read.
 * Limits: the scratch that moe_create_indices_workspace_size(num_slots,
 *   n_experts) reports must fit in MOE_NO_ALLOC_SCRATCH_BYTES; a larger
 *   request returns MOE_ERR_WORKSPACE before anything is enqueued. With 1 MiB
 *   the largest accepted num_slots is 2,076,672 over 128 experts, 1,040,384
 *   over 256 experts and 258,048 over 1024 experts (2^20 slots over 256
 *   experts need 1,053,952 bytes and are refused).
 * Allocation: the call makes no cudaMalloc, cudaFree or other allocating
 *   call. The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) and caches it, so make that first call before
 *   any stream capture begins. The cached address is not looked up again:
 *   do not reset the device (cudaDeviceReset) or otherwise destroy and
 *   recreate its primary context while the process still calls this entry
 *   point.
 * Sharing: all calls on a device use the same array. Calls whose work
 *   overlaps on the GPU (different streams, no ordering between them) race on
 *   it and give wrong results. Calls ordered one after another are safe.
 *   No scratch word needs clearing between calls: each call writes every
 *   word it reads before reading it.
 */
#define MOE_NO_ALLOC_SCRATCH_BYTES (1u << 20)
moe_status_t moe_create_indices_no_alloc(uint32_t* token_expert_order,
                                         uint32_t* expert_start_indices,
                                         uint32_t* restore_token_order, int32_t* expert_ids,
                                         uint32_t* expert_usage_stats, const int32_t* topk_ids,
                                         int64_t num_slots, int32_t n_experts,
                                         uint32_t* device_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTING_H */
