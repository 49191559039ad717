// Oracle for the MoE routing hot path (test infrastructure only; see moe_oracle.h).
//
// Written for clarity, not speed: each stage follows its definition step by
// step, with std::sort / std::fma as the only library primitives.
#include "moe_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

namespace {

float bf16_bits_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// exp(x) for the sigmoid score loader, in fp32, following Cody and Waite's
// range reduction ("Software Manual for the Elementary Functions", 1980):
//   clamp x to [-87, 88];  n = round-to-nearest-even(x * log2(e));
//   r = (x - n * ln2_head) - n * ln2_tail   (two fused multiply-adds; ln2_head
//       = 0.693145751953125 has 12 trailing zero bits, ln2_tail = ln2 - head);
//   exp(r) = sum_{k=0..7} r^k / k!   (Horner's rule, fused multiply-adds);
//   exp(x) = exp(r) * 2^n.
float exp_cody_waite(float x) {
  x = std::fmin(std::fmax(x, -87.0f), 88.0f);
  const float n = std::rint(x * 1.44269504088896341f);
  float r = std::fma(-n, 0.693145751953125f, x);
  r = std::fma(-n, 1.42860682030941723e-6f, r);
  const float inv_fact[8] = {1.0f, 1.0f, 0.5f, 1.66666666666666667e-1f, 4.16666666666666667e-2f,
                             8.33333333333333333e-3f, 1.38888888888888889e-3f,
                             1.98412698412698413e-4f};
  float p = inv_fact[7];
  for (int k = 6; k >= 0; --k) p = std::fma(p, r, inv_fact[k]);
  return p * std::ldexp(1.0f, static_cast<int>(n));
}

}  // namespace

// The exp that both score loaders below use, one value per element (its
// own pin compares it with a double-precision exp).
extern "C" int oracle_exp(const float* x, int64_t n, float* out) {
  if (n < 0) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) {
    if (std::isnan(x[i])) return ORACLE_ERR_NAN;
    out[i] = exp_cody_waite(x[i]);
  }
  return ORACLE_OK;
}

// group_limited_router_kernel, Parameters scores_input_fn: an optional loader
// of each (token, expert) score; here the score of a gate logit x is its
// sigmoid 1 / (1 + exp(-x)).
extern "C" int oracle_sigmoid(const float* x, int64_t n, float* out) {
  if (n < 0) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) {
    if (std::isnan(x[i])) return ORACLE_ERR_NAN;
    out[i] = 1.0f / (1.0f + exp_cody_waite(-x[i]));
  }
  return ORACLE_OK;
}

// group_limited_router_kernel, Parameters scores_input_fn: here the scores of
// one token's gate logits x[0..E) are their softmax, exp(x_e - max x) divided
// by the sum of those exponentials; the sum is taken in ascending expert
// order. All in fp32 with the exp above.
extern "C" int oracle_softmax(const float* x, int64_t rows, int32_t cols, float* out) {
  if (rows < 0 || cols <= 0) return ORACLE_ERR_ARG;
  std::vector<float> ex(cols);
  for (int64_t r = 0; r < rows; ++r) {
    const float* row = x + r * cols;
    float m = row[0];
    for (int32_t e = 0; e < cols; ++e) {
      if (std::isnan(row[e])) return ORACLE_ERR_NAN;
      if (row[e] > m) m = row[e];
    }
    float sum = 0.0f;
    for (int32_t e = 0; e < cols; ++e) {
      ex[e] = exp_cody_waite(row[e] - m);
      sum += ex[e];
    }
    for (int32_t e = 0; e < cols; ++e) out[r * cols + e] = ex[e] / sum;
  }
  return ORACLE_OK;
}

// group_limited_router_kernel, description paragraph: experts are split into
// n_groups groups, the topk_group best groups are kept, and the
// n_experts_per_tok experts are chosen from the kept groups; the bias is added
// for the selection only. Parameters norm_weights and Args
// routed_scaling_factor: the chosen weights are optionally normalised to sum
// to one, then multiplied by the factor. Args expert_weights: the weights are
// the scores without the bias.
extern "C" int oracle_route(const float* scores, const float* bias, int64_t T, int32_t E,
                            int32_t K, int32_t n_groups, int32_t topk_group,
                            int32_t norm_weights, float scale, int32_t* ids_out,
                            float* w_out) {
  if (T < 0 || E <= 0 || n_groups <= 0 || E % n_groups != 0) return ORACLE_ERR_ARG;
  const int32_t S = E / n_groups;  // experts per group
  if (topk_group <= 0 || topk_group > n_groups) return ORACLE_ERR_ARG;
  if (K <= 0 || K > topk_group * S) return ORACLE_ERR_ARG;

  std::vector<float> b(E);
  std::vector<float> g(n_groups);
  std::vector<int32_t> group_order(n_groups);
  std::vector<int32_t> allowed;
  std::vector<float> group_vals;

  for (int64_t t = 0; t < T; ++t) {
    const float* s = scores + t * E;

    // Step 1: biased selection score, fp32.
    for (int32_t e = 0; e < E; ++e) {
      if (std::isnan(s[e]) || std::isnan(bias[e])) return ORACLE_ERR_NAN;
      b[e] = s[e] + bias[e];
    }

    // Step 2: group score = top-1 + top-2 of the group's biased scores.
    for (int32_t j = 0; j < n_groups; ++j) {
      group_vals.assign(b.begin() + j * S, b.begin() + (j + 1) * S);
      std::sort(group_vals.begin(), group_vals.end(), [](float x, float y) { return x > y; });
      g[j] = (S == 1) ? group_vals[0] : group_vals[0] + group_vals[1];
    }

    // Step 3: the topk_group groups with the highest scores, ties to the lower index.
    for (int32_t j = 0; j < n_groups; ++j) group_order[j] = j;
    std::sort(group_order.begin(), group_order.end(), [&](int32_t x, int32_t y) {
      if (g[x] != g[y]) return g[x] > g[y];
      return x < y;
    });

    // Step 4: experts of the kept groups, ranked by biased score, ties to the lower index.
    allowed.clear();
    for (int32_t m = 0; m < topk_group; ++m) {
      const int32_t j = group_order[m];
      for (int32_t e = j * S; e < (j + 1) * S; ++e) allowed.push_back(e);
    }
    std::sort(allowed.begin(), allowed.end(), [&](int32_t x, int32_t y) {
      if (b[x] != b[y]) return b[x] > b[y];
      return x < y;
    });

    // Step 5: weights from the unbiased scores; optional normalisation, then scaling.
    int32_t* ids = ids_out + t * K;
    float* w = w_out + t * K;
    for (int32_t k = 0; k < K; ++k) {
      ids[k] = allowed[k];
      w[k] = s[allowed[k]];
    }
    if (norm_weights) {
      float sum = 0.0f;
      for (int32_t k = 0; k < K; ++k) sum = sum + w[k];
      for (int32_t k = 0; k < K; ++k) w[k] = w[k] / sum;
    }
    for (int32_t k = 0; k < K; ++k) w[k] = w[k] * scale;
  }
  return ORACLE_OK;
}

// moe_create_indices, description paragraph: a bucket sort of the flat
// topk_ids by expert. Args: token_expert_order lists slot indices grouped by
// expert, expert_start_indices are CSR start offsets, restore_token_order maps
// each slot to its position in token_expert_order, expert_ids lists the
// active experts, expert_usage_stats = [max tokens per expert, active experts].
extern "C" int oracle_create_indices(const int32_t* topk_ids, int64_t N, int32_t E,
                                     uint32_t* token_expert_order,
                                     uint32_t* expert_start_indices,
                                     uint32_t* restore_token_order, int32_t* expert_ids,
                                     uint32_t* expert_usage_stats) {
  if (N < 0 || E <= 0 || N > 0xFFFFFFFFll) return ORACLE_ERR_ARG;
  std::vector<uint32_t> count(E, 0);
  for (int64_t i = 0; i < N; ++i) {
    if (topk_ids[i] < 0 || topk_ids[i] >= E) return ORACLE_ERR_DATA;
    count[topk_ids[i]] += 1;
  }

  // Active experts in ascending id, with their start offsets.
  std::vector<uint32_t> cursor(E, 0);
  uint32_t offset = 0, active = 0, max_count = 0;
  for (int32_t e = 0; e < E; ++e) {
    max_count = std::max(max_count, count[e]);
    if (count[e] == 0) continue;
    expert_ids[active] = e;
    expert_start_indices[active] = offset;
    cursor[e] = offset;
    offset += count[e];
    active += 1;
  }
  for (uint32_t j = active; j <= static_cast<uint32_t>(E); ++j)
    expert_start_indices[j] = static_cast<uint32_t>(N);
  for (uint32_t j = active; j < static_cast<uint32_t>(E); ++j) expert_ids[j] = -1;

  // One pass in slot order places each slot at its expert's cursor: stable by construction.
  for (int64_t i = 0; i < N; ++i) {
    const uint32_t pos = cursor[topk_ids[i]]++;
    token_expert_order[pos] = static_cast<uint32_t>(i);
    restore_token_order[i] = pos;
  }

  expert_usage_stats[0] = max_count;
  expert_usage_stats[1] = active;
  return ORACLE_OK;
}

// moe_create_indices, Args scales_offset_p: aligned scale offsets for an
// FP8/block-scaled grouped matmul. Reading (the page gives no alignment): each
// active expert's rows are padded to a multiple of row_align, and the offsets
// are the running sums of the padded counts, in active-expert order.
extern "C" int oracle_scales_offsets(const int32_t* topk_ids, int64_t N, int32_t E,
                                     uint32_t row_align, uint32_t* out) {
  if (N < 0 || E <= 0 || row_align == 0) return ORACLE_ERR_ARG;
  std::vector<uint64_t> count(E, 0);
  for (int64_t i = 0; i < N; ++i) {
    if (topk_ids[i] < 0 || topk_ids[i] >= E) return ORACLE_ERR_DATA;
    count[topk_ids[i]] += 1;
  }
  uint64_t offset = 0;
  int32_t j = 0;
  for (int32_t e = 0; e < E; ++e) {
    if (count[e] == 0) continue;
    out[j++] = static_cast<uint32_t>(offset);
    offset += (count[e] + row_align - 1) / row_align * row_align;
  }
  for (; j <= E; ++j) out[j] = static_cast<uint32_t>(offset);
  return ORACLE_OK;
}

// moe_finalize, description paragraph: each output element gathers its
// token's K rows of down through restore_order, scales each by its router
// weight and sums in fp32 (Args: output, down, restore_order, router_weight).
static int finalize_one_token(const uint16_t* down, const uint32_t* restore, const float* w,
                              int64_t T, int32_t K, int64_t H, int64_t t, float* out_row) {
  const int64_t N = T * K;
  for (int32_t k = 0; k < K; ++k)
    if (static_cast<int64_t>(restore[t * K + k]) >= N) return ORACLE_ERR_DATA;
  for (int64_t h = 0; h < H; ++h) {
    float acc = 0.0f;
    for (int32_t k = 0; k < K; ++k) {
      const int64_t row = restore[t * K + k];
      acc = std::fma(w[t * K + k], bf16_bits_to_float(down[row * H + h]), acc);
    }
    out_row[h] = acc;
  }
  return ORACLE_OK;
}

extern "C" int oracle_finalize(const uint16_t* down, const uint32_t* restore, const float* w,
                               int64_t T, int32_t K, int64_t H, float* out) {
  if (T < 0 || K <= 0 || H < 0) return ORACLE_ERR_ARG;
  for (int64_t t = 0; t < T; ++t) {
    int rc = finalize_one_token(down, restore, w, T, K, H, t, out + t * H);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}

extern "C" int oracle_finalize_tokens(const uint16_t* down, const uint32_t* restore,
                                      const float* w, int64_t T, int32_t K, int64_t H,
                                      const int64_t* tokens, int64_t n_sel, float* out) {
  if (T < 0 || K <= 0 || H < 0 || n_sel < 0) return ORACLE_ERR_ARG;
  for (int64_t j = 0; j < n_sel; ++j) {
    if (tokens[j] < 0 || tokens[j] >= T) return ORACLE_ERR_ARG;
    int rc = finalize_one_token(down, restore, w, T, K, H, tokens[j], out + j * H);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}

extern "C" int oracle_finalize_f64(const uint16_t* down, const uint32_t* restore, const float* w,
                                   int64_t T, int32_t K, int64_t H, double* out) {
  if (T < 0 || K <= 0 || H < 0) return ORACLE_ERR_ARG;
  const int64_t N = T * K;
  for (int64_t t = 0; t < T; ++t) {
    for (int32_t k = 0; k < K; ++k)
      if (static_cast<int64_t>(restore[t * K + k]) >= N) return ORACLE_ERR_DATA;
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int32_t k = 0; k < K; ++k) {
        const int64_t row = restore[t * K + k];
        acc += static_cast<double>(w[t * K + k]) *
               static_cast<double>(bf16_bits_to_float(down[row * H + h]));
      }
      out[t * H + h] = acc;
    }
  }
  return ORACLE_OK;
}

// moe_create_indices, description paragraph: slots are grouped by expert so
// that downstream kernels such as the grouped matmul process each expert's
// tokens contiguously. Row p of that expert-contiguous input is the row of the
// token owning slot token_expert_order[p] (slot i = t*K + k belongs to t).
extern "C" int oracle_permute(const uint16_t* input, const uint32_t* token_expert_order,
                              int64_t T, int32_t K, int64_t H, uint16_t* out) {
  if (T < 0 || K <= 0 || H < 0) return ORACLE_ERR_ARG;
  const int64_t N = T * K;
  for (int64_t p = 0; p < N; ++p) {
    const int64_t slot = token_expert_order[p];
    if (slot >= N) return ORACLE_ERR_DATA;
    const int64_t t = slot / K;
    for (int64_t h = 0; h < H; ++h) out[p * H + h] = input[t * H + h];
  }
  return ORACLE_OK;
}
