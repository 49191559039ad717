/*
 * Oracle for the MoE routing hot path: a plain, slow, single-threaded CPU
 * restatement of what the three stages compute.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. It shares no code, header,
 * table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Sources (Mojo kernel library API pages):
 *   - "group_limited_router_kernel": description paragraph; Parameters
 *     (n_groups, topk_group, norm_weights); Args (expert_indices,
 *     expert_weights, expert_bias, routed_scaling_factor).
 *   - "moe_create_indices": description paragraph; Args (token_expert_order,
 *     expert_start_indices, restore_token_order, expert_ids,
 *     expert_usage_stats, topk_ids).
 *   - "moe_finalize": description paragraph; Args (output, down,
 *     restore_order, router_weight).
 *   - "group_limited_router_kernel", Parameters scores_input_fn: sigmoid and
 *     softmax score loaders for gate logits;
 *   - the expert-contiguous token rows that the grouped matmul consumes
 *     ("moe_create_indices", description paragraph).
 *
 * Readings where the pages are silent:
 *   - group score = sum of the group's two largest biased scores (one score if
 *     the group has a single expert);
 *   - ties (groups and experts) go to the lower index, comparing IEEE values;
 *   - expert_indices rows are in selection order (biased score descending,
 *     ties to the lower index);
 *   - the normalisation sum runs sequentially in that order, in fp32, with no
 *     epsilon;
 *   - "token index" in token_expert_order is the flat slot i = t*K + k, and
 *     order within one expert is ascending i;
 *   - expert_start_indices is a compact CSR over the active experts in
 *     ascending id: entries 0..A are the starts plus the end (= N), entries
 *     A+1..E are N; expert_ids[j] = -1 for j >= A;
 *   - finalize accumulates k = 0..K-1 in order with fp32 fused multiply-add
 *     from 0.0f; the comparison with bf16 outputs happens before rounding.
 *
 * Parity pins: route selection is pinned by brute-force subset enumeration,
 * a library top-k and tie-stress inputs; the index by a library stable sort
 * and the inverse-permutation / CSR invariants; finalize by closed forms, a
 * library gather-and-sum and the fp64 variant below.
 *
 * All functions return 0 on success and a negative code on invalid input.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_NAN -2
#define ORACLE_ERR_DATA -3

/* The exp of the score loaders, exposed for its own pin: out[i] =
 * exp(clamp(x[i], -87, 88)) in fp32 by Cody-Waite reduction and a degree-7
 * Taylor polynomial (see the .cpp). */
int oracle_exp(const float* x, int64_t n, float* out);

/* Sigmoid score loader: out[i] = 1 / (1 + exp(-x[i])) in fp32, with the exp
 * of oracle_exp. */
int oracle_sigmoid(const float* x, int64_t n, float* out);

/* Softmax score loader (Parameters scores_input_fn): out[r, e] =
 * exp(x[r, e] - max_e' x[r, e']) / sum_e' exp(x[r, e'] - max), fp32, the sum
 * in ascending e, exp as for oracle_sigmoid. */
int oracle_softmax(const float* x, int64_t rows, int32_t cols, float* out);

/* Router. scores [T,E] fp32 row-major, bias [E] fp32.
 * ids_out [T,K] int32, w_out [T,K] fp32. */
int oracle_route(const float* scores, const float* bias, int64_t T, int32_t E, int32_t K,
                 int32_t n_groups, int32_t topk_group, int32_t norm_weights, float scale,
                 int32_t* ids_out, float* w_out);

/* Index builder over N flat slots. topk_ids [N] int32 in [0,E).
 * token_expert_order [N], expert_start_indices [E+1], restore_token_order [N],
 * expert_ids [E], expert_usage_stats [2]. */
int oracle_create_indices(const int32_t* topk_ids, int64_t N, int32_t E,
                          uint32_t* token_expert_order, uint32_t* expert_start_indices,
                          uint32_t* restore_token_order, int32_t* expert_ids,
                          uint32_t* expert_usage_stats);

/* Aligned scale offsets of the active experts for a block-scaled grouped
 * matmul: out [E+1], entry j < A = sum over active experts j' < j of the
 * expert's slot count rounded up to a multiple of `row_align`; entries A..E =
 * the padded total. */
int oracle_scales_offsets(const int32_t* topk_ids, int64_t N, int32_t E, uint32_t row_align,
                          uint32_t* out);

/* Finalize, fp32 accumulation, result before bf16 rounding.
 * down [T*K, H] bf16 bit patterns, restore [T*K], w [T,K], out [T,H] fp32. */
int oracle_finalize(const uint16_t* down, const uint32_t* restore, const float* w, int64_t T,
                    int32_t K, int64_t H, float* out);

/* Same, for the listed tokens only: out [n_sel, H] fp32 (row j = token tokens[j]). */
int oracle_finalize_tokens(const uint16_t* down, const uint32_t* restore, const float* w,
                           int64_t T, int32_t K, int64_t H, const int64_t* tokens,
                           int64_t n_sel, float* out);

/* Expert-contiguous token rows: out [T*K, H] row p = input row token_expert_order[p] / K.
 * input [T, H] and out hold bf16 bit patterns. */
int oracle_permute(const uint16_t* input, const uint32_t* token_expert_order, int64_t T, int32_t K,
                   int64_t H, uint16_t* out);

/* fp64 accumulation of the same sum (bounds the fp32 oracle's own rounding). */
int oracle_finalize_f64(const uint16_t* down, const uint32_t* restore, const float* w, int64_t T,
                        int32_t K, int64_t H, double* out);

#ifdef __cplusplus
}
#endif

#endif
