// Device code of the group-limited top-k router, shared by the stand-alone
// router kernels and the fused router + index kernel.
//
// Page "group_limited_router_kernel", description paragraph: experts are split
// into n_groups groups, the topk_group best groups are kept and the
// n_experts_per_tok experts are chosen from them; the bias is added for the
// selection only (Args expert_bias, expert_weights); Parameters norm_weights
// and Args routed_scaling_factor fix the weight post-processing.
#pragma once

#include <math_constants.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;

// With at most 32 groups and C experts per lane, a group always spans at
// least one whole lane, so two layouts cover every shape.
enum GroupMode : int {
  kGroupsAllKept = 0,  // topk_group == n_groups: no group selection
  kGroupsSegment = 1,  // a group spans a power-of-two run of whole lanes
  kGroupsGeneric = 2   // anything else: group scores through shared memory
};

struct RouteArgs {
  int32_t* ids;
  float* weights;
  const float* scores;
  const float* bias;
  int64_t T;
  int E, K, G, M, S;
  int norm;
  float scale;
  int group_mode;
  int seg_lanes;  // lanes per group in kGroupsSegment
  int score_fn;   // moe_score_fn_t applied to every loaded score
  // Warp path: floats of shared memory per warp: E for the generic group
  // layout's biased scores, then E for the token's softmax scores.
  int warp_smem_words;
  int softmax_off;
  // Segment layout: an expert's selection key keeps the top 32 - key_bits
  // bits of its order key and carries key_low - e in the low key_bits bits
  // (key_low = 2^key_bits - 1, key_bits = bits of E - 1).
  int key_bits;
  uint32_t key_low;
};

// exp(x) in fp32 by Cody-Waite range reduction (W. J. Cody and W. Waite,
// "Software Manual for the Elementary Functions", 1980): x = n ln2 + r with
// |r| <= ln2/2, ln2 split into a head with 12 trailing zero bits (so n*head is
// exact) and a tail; exp(r) by its Taylor series to degree 7 in Horner form
// with fused multiply-adds; 2^n assembled from exponent bits. x is clamped to
// [-87, 88] so that 2^n is a normal float. Every step is a correctly rounded
// fp32 operation, so the result is reproducible bit for bit.
__device__ __forceinline__ float score_exp_f32(float x) {
  x = fminf(fmaxf(x, -87.0f), 88.0f);
  const float n = rintf(__fmul_rn(x, 1.44269504088896341f));
  float r = __fmaf_rn(-n, 0.693145751953125f, x);
  r = __fmaf_rn(-n, 1.42860682030941723e-6f, r);
  float p = 1.98412698412698413e-4f;             // 1/7!
  p = __fmaf_rn(p, r, 1.38888888888888889e-3f);  // 1/6!
  p = __fmaf_rn(p, r, 8.33333333333333333e-3f);  // 1/5!
  p = __fmaf_rn(p, r, 4.16666666666666667e-2f);  // 1/4!
  p = __fmaf_rn(p, r, 1.66666666666666667e-1f);  // 1/3!
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  return __fmul_rn(p, __int_as_float(((int)n + 127) << 23));
}

// The page's scores_input_fn for the element-wise loaders: the score of
// (token, expert) from the loaded value.
__device__ __forceinline__ float apply_score_fn(int fn, float x) {
  if (fn == MOE_SCORES_SIGMOID) return __fdiv_rn(1.0f, __fadd_rn(1.0f, score_exp_f32(-x)));
  return x;
}

// Running top-2 of a stream of values (multiset: equal values both count).
__device__ __forceinline__ void top2_push(float& t1, float& t2, float x) {
  t2 = fmaxf(t2, fminf(t1, x));
  t1 = fmaxf(t1, x);
}

// Rank groups by (score desc, index asc) and return the bit mask of the M best.
// Lane j < G holds g_j on entry.
__device__ __forceinline__ uint32_t keep_best_groups(float gj, int lane, int G, int M) {
  int ahead = 0;
#pragma unroll 8
  for (int j = 0; j < G; ++j) {
    const float gx = __shfl_sync(kFullMask, gj, j);
    ahead += (gx > gj) || (gx == gj && j < lane);
  }
  return __ballot_sync(kFullMask, lane < G && ahead < M);
}

// The C scores of row t that lane l owns (experts l*C .. l*C+C-1).
template <int C, bool kVec>
__device__ __forceinline__ void load_lane_scores(const RouteArgs& a, int64_t t, int e0,
                                                 const bool (&valid)[C], float (&s)[C]) {
  const float* row = a.scores + t * a.E;
  if constexpr (kVec) {
#pragma unroll
    for (int q = 0; q < C / 4; ++q) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e0 + 4 * q < a.E) v = __ldg(reinterpret_cast<const float4*>(row + e0 + 4 * q));
      s[4 * q + 0] = v.x;
      s[4 * q + 1] = v.y;
      s[4 * q + 2] = v.z;
      s[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int c = 0; c < C; ++c) s[c] = valid[c] ? __ldg(row + e0 + c) : 0.0f;
  }
}

// Exact top-K by K rounds of a warp-wide max over each lane's best key; the
// winning lane recomputes its best from all of its keys. Returns, in lane r <
// K, the expert chosen in round r.
template <int C>
__device__ __forceinline__ int select_by_full_rounds(uint32_t (&key)[C], int lane, int e0, int K) {
  uint32_t head = 0;
  int head_pos = 0;
#pragma unroll
  for (int c = 0; c < C; ++c)
    if (key[c] > head) { head = key[c]; head_pos = c; }
  int my_id = 0;
  for (int r = 0; r < K; ++r) {
    const uint32_t best = __reduce_max_sync(kFullMask, head);
    const unsigned holders = __ballot_sync(kFullMask, head == best && head != 0u);
    const int win_lane = holders ? __ffs(holders) - 1 : 0;
    const int id = __shfl_sync(kFullMask, e0 + head_pos, win_lane);
    if (lane == r) my_id = id;
    if (lane == win_lane) {
#pragma unroll
      for (int c = 0; c < C; ++c)
        if (c == head_pos) key[c] = 0u;
      head = 0;
      head_pos = 0;
#pragma unroll
      for (int c = 0; c < C; ++c)
        if (key[c] > head) { head = key[c]; head_pos = c; }
    }
  }
  return my_id;
}

// The softmax loader on one token's logits, held C per lane (lane l: experts
// l*C .. l*C+C-1): s := exp(s - max) / sum, with the sum taken in ascending
// expert order (each lane adds its experts to the running sum of the lanes
// before it), so the result is bit-identical to a sequential loop. The scores
// are also left in `strip` (E floats) for the weights.
template <int C>
__device__ __forceinline__ void softmax_lane_row(const RouteArgs& a, float (&s)[C],
                                                 const bool (&valid)[C], int lane, int e0,
                                                 float* strip) {
  float m = -CUDART_INF_F;
#pragma unroll
  for (int c = 0; c < C; ++c)
    if (valid[c]) m = fmaxf(m, s[c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, off));
  float ex[C];
#pragma unroll
  for (int c = 0; c < C; ++c) ex[c] = valid[c] ? score_exp_f32(__fsub_rn(s[c], m)) : 0.0f;
  const int lanes = (a.E + C - 1) / C;
  float run = 0.0f;
  for (int l = 0; l < lanes; ++l) {
    if (lane == l) {
#pragma unroll
      for (int c = 0; c < C; ++c)
        if (valid[c]) run = __fadd_rn(run, ex[c]);
    }
    run = __shfl_sync(kFullMask, run, l);
  }
  __syncwarp();  // the previous token's weights have been read from the strip
#pragma unroll
  for (int c = 0; c < C; ++c) {
    s[c] = valid[c] ? __fdiv_rn(ex[c], run) : 0.0f;
    if (valid[c]) strip[e0 + c] = s[c];
  }
  __syncwarp();
}

// Routes tokens first, first + stride, ... (below end) with the calling warp.
// Lane l holds experts l*C .. l*C+C-1. `warp_smem` is this warp's
// a.warp_smem_words floats of shared memory (the generic group layout's
// biased scores, the softmax loader's scores). After token t's ids and
// weights are written, lane k < K calls on_id(t, k, id). kSoftmax selects the
// softmax loader (a separate instantiation keeps the other loaders' register
// budget).
template <int C, bool kVec, bool kSoftmax, typename OnId>
__device__ __forceinline__ void route_tokens_warp(const RouteArgs& a, int64_t first, int64_t end,
                                                  int64_t stride, float* warp_smem,
                                                  OnId on_id) {
  static_assert(C >= 2, "the warp path holds at least two experts per lane");

  const int lane = threadIdx.x & 31;
  const int e0 = lane * C;

  float bias_r[C];
  bool valid[C];
  int n_valid = 0;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int e = e0 + c;
    valid[c] = e < a.E;
    bias_r[c] = valid[c] ? a.bias[e] : 0.0f;
    n_valid += valid[c];
  }
  // In the segment layout a lane's experts all belong to one group.
  const int lane_grp = n_valid > 0 ? e0 / a.S : 31;

  float s_next[C];
  if (first < end) load_lane_scores<C, kVec>(a, first, e0, valid, s_next);

  for (int64_t t = first; t < end; t += stride) {
    float s[C];
#pragma unroll
    for (int c = 0; c < C; ++c) s[c] = s_next[c];
    if (t + stride < end) load_lane_scores<C, kVec>(a, t + stride, e0, valid, s_next);
    if constexpr (kSoftmax) {
      softmax_lane_row<C>(a, s, valid, lane, e0, warp_smem + a.softmax_off);
    } else if (a.score_fn != MOE_SCORES_AS_GIVEN) {
#pragma unroll
      for (int c = 0; c < C; ++c) s[c] = apply_score_fn(a.score_fn, s[c]);
    }

    float b[C];
#pragma unroll
    for (int c = 0; c < C; ++c) b[c] = valid[c] ? __fadd_rn(s[c], bias_r[c]) : -CUDART_INF_F;

    int my_id = 0;
    if (a.group_mode == kGroupsGeneric) {
      // ---- groups through shared memory, then the exact full-round selection ----
      float* wb = warp_smem;
#pragma unroll
      for (int c = 0; c < C; ++c)
        if (valid[c]) wb[e0 + c] = b[c];
      __syncwarp();
      float gj = 0.0f;
      if (lane < a.G) {
        float t1 = -CUDART_INF_F, t2 = -CUDART_INF_F;
        for (int e = lane * a.S; e < (lane + 1) * a.S; ++e) top2_push(t1, t2, wb[e]);
        gj = (a.S == 1) ? t1 : __fadd_rn(t1, t2);
      }
      __syncwarp();
      const uint32_t kept = keep_best_groups(gj, lane, a.G, a.M);
      uint32_t key[C];
#pragma unroll
      for (int c = 0; c < C; ++c)
        key[c] = (valid[c] && ((kept >> ((e0 + c) / a.S)) & 1u)) ? ordered_key(b[c]) : 0u;
      my_id = select_by_full_rounds<C>(key, lane, e0, a.K);
    } else {
      // ---- lane cache: the D best biased scores and their positions ----
      // (ties keep the lower position, so equal entries come in expert order)
      constexpr int D = C >= 3 ? 3 : 2;
      float v[D];
      int p[D];
#pragma unroll
      for (int j = 0; j < D; ++j) {
        v[j] = 0.0f;
        p[j] = 0;
      }
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const float x = b[c];
        bool g[D];
#pragma unroll
        for (int j = 0; j < D; ++j) g[j] = (j >= c) || x > v[j];  // empty slots take x
#pragma unroll
        for (int j = D - 1; j >= 1; --j) {
          if (j > c) continue;
          v[j] = g[j - 1] ? v[j - 1] : (g[j] ? x : v[j]);
          p[j] = g[j - 1] ? p[j - 1] : (g[j] ? c : p[j]);
        }
        v[0] = g[0] ? x : v[0];
        p[0] = g[0] ? c : p[0];
      }

      // ---- group selection (segment layout: the group's top-2 over its lanes) ----
      bool lane_allowed = n_valid > 0;
      if (a.group_mode == kGroupsSegment) {
        float t1 = n_valid > 0 ? v[0] : -CUDART_INF_F, t2 = n_valid > 0 ? v[1] : -CUDART_INF_F;
        for (int off = 1; off < a.seg_lanes; off <<= 1) {
          const float o1 = __shfl_xor_sync(kFullMask, t1, off);
          const float o2 = __shfl_xor_sync(kFullMask, t2, off);
          t2 = fmaxf(fminf(t1, o1), fmaxf(t2, o2));
          t1 = fmaxf(t1, o1);
        }
        const float g = __fadd_rn(t1, t2);
        const float gj = __shfl_sync(kFullMask, g, lane < a.G ? lane * a.seg_lanes : 0);
        const uint32_t kept = keep_best_groups(gj, lane, a.G, a.M);
        lane_allowed = lane_allowed && ((kept >> lane_grp) & 1u);
      }
      const int n_allowed = lane_allowed ? n_valid : 0;

      // ---- K rounds of a warp-wide max over the cached heads ----
      uint32_t k[D];
      int id[D];
#pragma unroll
      for (int j = 0; j < D; ++j) {
        k[j] = n_allowed > j ? ordered_key(v[j]) : 0u;
        id[j] = e0 + p[j];
      }
      int wins = 0;
      uint32_t kth = 0;
      int kth_id = 0;
#pragma unroll 8
      for (int r = 0; r < a.K; ++r) {
        const uint32_t best = __reduce_max_sync(kFullMask, k[0]);
        const unsigned holders = __ballot_sync(kFullMask, k[0] == best);
        const int win_lane = __ffs(holders) - 1;
        const int win_id = __shfl_sync(kFullMask, id[0], win_lane);
        if (lane == r) my_id = win_id;
        kth = best;
        kth_id = win_id;
        if (lane == win_lane) {
#pragma unroll
          for (int j = 0; j + 1 < D; ++j) {
            k[j] = k[j + 1];
            id[j] = id[j + 1];
          }
          k[D - 1] = 0u;
          ++wins;
        }
      }

      // ---- exactness check: a lane that gave up all D cached entries may hold
      // a further candidate that should have won a later round ----
      const bool needs_more = wins == D && n_allowed > D;
      if (__any_sync(kFullMask, needs_more) || kth == 0u) {
        float vn = -CUDART_INF_F;
        int cn = -1;
#pragma unroll
        for (int c = 0; c < C; ++c) {
          bool cached = false;
#pragma unroll
          for (int j = 0; j < D; ++j) cached = cached || c == p[j];
          if (valid[c] && !cached && (cn < 0 || b[c] > vn)) { vn = b[c]; cn = c; }
        }
        const uint32_t kn = ordered_key(vn);
        const bool beats = kn > kth || (kn == kth && e0 + cn < kth_id);
        if (kth == 0u || __any_sync(kFullMask, needs_more && beats)) {
          uint32_t key[C];
#pragma unroll
          for (int c = 0; c < C; ++c) key[c] = (valid[c] && lane_allowed) ? ordered_key(b[c]) : 0u;
          my_id = select_by_full_rounds<C>(key, lane, e0, a.K);
        }
      }
    }

    // ---- weights: unbiased score, optional normalisation, scaling ----
    const float* row = a.scores + t * a.E;
    float w = 0.0f;
    if (lane < a.K) {
      if constexpr (kSoftmax)  // (an id outside [0, E) is possible only for NaN scores)
        w = (unsigned)my_id < (unsigned)a.E ? warp_smem[a.softmax_off + my_id] : 0.0f;
      else
        w = apply_score_fn(a.score_fn, __ldg(row + my_id));
    }
    if (a.norm) {
      float sum = 0.0f;
#pragma unroll 8
      for (int k = 0; k < a.K; ++k) sum = __fadd_rn(sum, __shfl_sync(kFullMask, w, k));
      w = __fdiv_rn(w, sum);
    }
    w = __fmul_rn(w, a.scale);
    if (lane < a.K) {
      a.ids[t * a.K + lane] = my_id;
      a.weights[t * a.K + lane] = w;
      on_id(t, lane, my_id);
    }
  }
}


// ---------------------------------------------------------------- segment layout
// E = 32*L experts (L = 2 .. 32, a power of two), K <= 8: a segment of L lanes
// routes one token, so a warp routes 32/L tokens at once; lane j of a segment
// holds experts 32j .. 32j+31. Every expert gets a 32-bit selection key: the
// order key of its biased score with the low key_bits bits replaced by key_low
// - e. The keys are unique and name their expert, and two keys whose order
// keys differ above bit key_bits compare as (score desc, expert asc). Each
// lane sorts its 32 keys into a top-8 with sorting networks of unsigned
// min/max, the segment merges its lanes' lists in log2(L) butterfly steps,
// and the first K of the merged list are the token's experts. This equals the
// exact selection whenever the first K+1 keys differ above bit key_bits: then
// every other candidate's order key is below all K chosen ones and the chosen
// ones keep their order. Otherwise (two near-equal scores at the top, about
// 0.4% of the tokens of the prefill workload) the segment ranks the few
// candidates that can still be chosen by their exact 64-bit keys, and only
// when that set is not known from the lanes' lists is the token routed again
// by the exact warp path.

constexpr int kSegKeys = 32;        // experts per lane
constexpr int kSegTop = 8;          // length of the sorted lists (K <= 8)
constexpr int kSegBiasStride = 36;  // shared-memory floats per lane block of bias
constexpr int kSegCand = 32;        // tie resolution: candidate keys per token

__device__ __forceinline__ void cmpx_desc(uint32_t& a, uint32_t& b) {
  const uint32_t hi = max(a, b);
  b = min(a, b);
  a = hi;
}

// Sorts 8 keys into descending order (Batcher's odd-even merge sort: 19
// comparators in 6 layers).
__device__ __forceinline__ void sort8_desc(uint32_t (&x)[8]) {
  cmpx_desc(x[0], x[1]); cmpx_desc(x[2], x[3]); cmpx_desc(x[4], x[5]); cmpx_desc(x[6], x[7]);
  cmpx_desc(x[0], x[2]); cmpx_desc(x[1], x[3]); cmpx_desc(x[4], x[6]); cmpx_desc(x[5], x[7]);
  cmpx_desc(x[1], x[2]); cmpx_desc(x[5], x[6]);
  cmpx_desc(x[0], x[4]); cmpx_desc(x[1], x[5]); cmpx_desc(x[2], x[6]); cmpx_desc(x[3], x[7]);
  cmpx_desc(x[2], x[4]); cmpx_desc(x[3], x[5]);
  cmpx_desc(x[1], x[2]); cmpx_desc(x[3], x[4]); cmpx_desc(x[5], x[6]);
}

// a := the 8 largest keys of the descending lists a and b, descending. The
// element-wise maximum of a and reversed b holds exactly those keys and is
// bitonic, so three half-cleaner layers sort it (K. E. Batcher, "Sorting
// networks and their applications", 1968).
__device__ __forceinline__ void merge8_desc(uint32_t (&a)[8], const uint32_t (&b)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = max(a[i], b[7 - i]);
  cmpx_desc(a[0], a[4]); cmpx_desc(a[1], a[5]); cmpx_desc(a[2], a[6]); cmpx_desc(a[3], a[7]);
  cmpx_desc(a[0], a[2]); cmpx_desc(a[1], a[3]); cmpx_desc(a[4], a[6]); cmpx_desc(a[5], a[7]);
  cmpx_desc(a[0], a[1]); cmpx_desc(a[2], a[3]); cmpx_desc(a[4], a[5]); cmpx_desc(a[6], a[7]);
}

// x[i] for a run-time i in [0, 8) without local memory.
__device__ __forceinline__ uint32_t pick8(const uint32_t (&x)[8], int i) {
  uint32_t r = x[0];
#pragma unroll
  for (int q = 1; q < 8; ++q) r = (i == q) ? x[q] : r;
  return r;
}

// Selection key of a biased score b that is not -0 (the staged bias holds no
// -0, and x + y is -0 only when both are -0), so the order key needs no
// zero fold.
template <uint32_t kKeyLow>
__device__ __forceinline__ uint32_t selection_key(float b, uint32_t tag) {
  const uint32_t u = __float_as_uint(b);
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return (k & ~kKeyLow) | tag;
}

// Index bits of the selection keys for E experts: the smallest b >= 1 with
// 2^b >= E. plan_route sets RouteArgs::key_bits with it, and the layouts that
// know E at compile time (segment, staged) use it as a constant.
__host__ __device__ constexpr int key_bits_for(int E) {
  int b = 1;
  while ((1 << b) < E) ++b;
  return b;
}

// The routing score of one expert from its loaded value x: the score
// function, or for the softmax loader exp(x - m) / sum with the row's max m
// and its sum in ascending expert order. These are the operations the whole
// row goes through, so the result has the same bits.
template <bool kSoftmax>
__device__ __forceinline__ float seg_score(const RouteArgs& a, float x, float m, float sum) {
  if constexpr (kSoftmax)
    return __fdiv_rn(score_exp_f32(__fsub_rn(x, m)), sum);
  else
    return apply_score_fn(a.score_fn, x);
}

// This lane's 32 loaded values of a row (16-byte loads).
__device__ __forceinline__ void load_seg_row(const float* row, float (&x)[kSegKeys]) {
#pragma unroll
  for (int q = 0; q < kSegKeys / 4; ++q) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(row) + q);
    x[4 * q + 0] = v.x;
    x[4 * q + 1] = v.y;
    x[4 * q + 2] = v.z;
    x[4 * q + 3] = v.w;
  }
}

// b := scores + bias, in place (b holds scores on entry).
__device__ __forceinline__ void add_seg_bias(const float* bias_j, float (&b)[kSegKeys]) {
#pragma unroll
  for (int q = 0; q < kSegKeys / 4; ++q) {
    const float4 c = *reinterpret_cast<const float4*>(bias_j + 4 * q);
    b[4 * q + 0] = __fadd_rn(b[4 * q + 0], c.x);
    b[4 * q + 1] = __fadd_rn(b[4 * q + 1], c.y);
    b[4 * q + 2] = __fadd_rn(b[4 * q + 2], c.z);
    b[4 * q + 3] = __fadd_rn(b[4 * q + 3], c.w);
  }
}

// Copies the bias into shared memory in the segment layout (call from warp
// 0, then __syncthreads): lane block j at s_bias + kSegBiasStride * j, so
// the eight 16-byte loads of a quarter warp hit distinct banks. A -0 bias is
// stored as +0: s + (-0) and s + (+0) differ only for s = -0, where they give
// -0 and +0, which compare equal, so no selection or group score changes and
// no biased score is ever -0. The loads are independent 16-byte loads (E is a
// multiple of 32 and the plan requires a 16-byte aligned bias).
__device__ __forceinline__ void stage_seg_bias(const RouteArgs& a, float* s_bias) {
  const int lane = threadIdx.x & 31;
  const float4* src = reinterpret_cast<const float4*>(a.bias);
  float4 v[MOE_MAX_EXPERTS / 128];
#pragma unroll
  for (int q = 0; q < MOE_MAX_EXPERTS / 128; ++q) {
    const int i = lane + 32 * q;  // float4 index: experts 4i .. 4i+3
    if (4 * i < a.E) v[q] = __ldg(src + i);
  }
#pragma unroll
  for (int q = 0; q < MOE_MAX_EXPERTS / 128; ++q) {
    const int i = lane + 32 * q;
    if (4 * i < a.E) {
      const int e = 4 * i;
      const float4 f = make_float4(__fadd_rn(v[q].x, 0.0f), __fadd_rn(v[q].y, 0.0f),
                                   __fadd_rn(v[q].z, 0.0f), __fadd_rn(v[q].w, 0.0f));
      *reinterpret_cast<float4*>(s_bias + kSegBiasStride * (e / kSegKeys) + e % kSegKeys) = f;
    }
  }
}

// The exact warp path for one token, out of line: it runs for few tokens, and
// keeping it out of the segment loop keeps that loop's code small.
template <int L, bool kSoftmax, typename OnId>
__device__ __noinline__ void route_one_token_exact(const RouteArgs a, int64_t t, float* warp_smem,
                                                   OnId on_id) {
  // (the warp path's vector loads need C = L to be a multiple of 4)
  route_tokens_warp<L, L % 4 == 0, kSoftmax>(a, t, t + 1, 1, warp_smem, on_id);
}

// Warps per CTA of a segment-layout launch: 8, or fewer when 8-warp CTAs
// would leave SMs without one (few tokens per warp-iteration count: 32/L
// tokens each).
inline int seg_warps_per_cta(int64_t T, int L, int sm_count) {
  const int64_t iters = (T + 32 / L - 1) / (32 / L);
  if (iters >= (int64_t)sm_count * kRouteWarps) return kRouteWarps;
  const int64_t w = (iters + 4 * (int64_t)sm_count - 1) / (4 * (int64_t)sm_count);
  return (int)(w < 1 ? 1 : w);
}

// Routes the tokens of warps warp_id, warp_id + num_warps, ... (32/L tokens
// each) with the calling warp; s_bias is the bias from stage_seg_bias, cand
// and slot this warp's (32/L) * kSegCand and (32/L) * kSegTop words of shared
// memory for resolving ties, warp_smem its a.warp_smem_words floats for the
// warp path's softmax strip. After token t's ids and weights are written,
// on_id(t, k, id) is called once per k < K. kGroups: topk_group < n_groups (a
// group spans L/G whole lanes). kSoftmax: the softmax loader, whose sum runs
// in ascending expert order by handing the running sum from lane to lane of
// the segment (the order of a sequential loop, so the same bits).
template <int L, bool kGroups, bool kSoftmax, typename OnId>
__device__ __forceinline__ void route_tokens_seg(const RouteArgs& a, const float* s_bias,
                                                 uint64_t* cand, int* slot, float* warp_smem,
                                                 int64_t warp_id, int64_t num_warps,
                                                 OnId on_id) {
  static_assert(L >= 2 && L <= 32 && (L & (L - 1)) == 0, "segments of 2 .. 32 lanes");
  constexpr int kTokens = 32 / L;                 // tokens per warp
  constexpr int kOut = (kSegTop + L - 1) / L;     // list entries a lane writes out
  const int lane = threadIdx.x & 31;
  const int j = lane & (L - 1);
  const int seg_base = lane & ~(L - 1);
  const unsigned seg_mask = (L == 32 ? kFullMask : ((1u << L) - 1u) << seg_base);
  const int e0 = kSegKeys * j;
  uint64_t* seg_cand = cand + (lane / L) * kSegCand;
  int* seg_slot = slot + (lane / L) * kSegTop;
  constexpr int kKeyBits = key_bits_for(kSegKeys * L);  // E = 32 * L here
  constexpr uint32_t kKeyLow = (1u << kKeyBits) - 1u;
  const uint32_t tag0 = kKeyLow - (uint32_t)e0;
  const int gl = kGroups ? L / a.G : L;  // lanes per group
  const int grp = j / gl;
  const float* bias_j = s_bias + kSegBiasStride * j;

  for (int64_t base = warp_id * kTokens; base < a.T; base += num_warps * kTokens) {
    const int64_t t = base + lane / L;
    const bool live = t < a.T;
    const float* row = a.scores + (live ? t : base) * a.E;

    // ---- selection keys, the group's top-2 and this lane's sorted top-8 ----
    uint32_t key[4][8];
    float t1 = -CUDART_INF_F, t2 = -CUDART_INF_F;
    float smax = 0.0f, ssum = 1.0f;  // the softmax loader's row max and sum
    {
      float b[kSegKeys];
      load_seg_row(row + e0, b);
      if constexpr (kSoftmax) {
        smax = -CUDART_INF_F;
#pragma unroll
        for (int i = 0; i < kSegKeys; ++i) smax = fmaxf(smax, b[i]);
#pragma unroll
        for (int off = 1; off < L; off <<= 1) smax = fmaxf(smax, __shfl_xor_sync(kFullMask, smax, off));
#pragma unroll
        for (int i = 0; i < kSegKeys; ++i) b[i] = score_exp_f32(__fsub_rn(b[i], smax));
        float run = 0.0f;
        for (int l = 0; l < L; ++l) {
          if (j == l) {
#pragma unroll
            for (int i = 0; i < kSegKeys; ++i) run = __fadd_rn(run, b[i]);
          }
          run = __shfl_sync(kFullMask, run, seg_base + l);
        }
        ssum = run;
#pragma unroll
        for (int i = 0; i < kSegKeys; ++i) b[i] = __fdiv_rn(b[i], ssum);
      } else if (a.score_fn != MOE_SCORES_AS_GIVEN) {
#pragma unroll
        for (int i = 0; i < kSegKeys; ++i) b[i] = apply_score_fn(a.score_fn, b[i]);
      }
      add_seg_bias(bias_j, b);
#pragma unroll
      for (int i = 0; i < kSegKeys; ++i) {
        key[i / 8][i % 8] = selection_key<kKeyLow>(b[i], tag0 - (uint32_t)i);
        if constexpr (kGroups) top2_push(t1, t2, b[i]);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) sort8_desc(key[q]);
    merge8_desc(key[0], key[1]);
    merge8_desc(key[2], key[3]);
    merge8_desc(key[0], key[2]);
    uint32_t (&mine)[8] = key[0];

    // ---- group selection: the group's top-2 sum ranked against the others ----
    if constexpr (kGroups) {
      for (int off = 1; off < gl; off <<= 1) {
        const float o1 = __shfl_xor_sync(kFullMask, t1, off);
        const float o2 = __shfl_xor_sync(kFullMask, t2, off);
        t2 = fmaxf(fminf(t1, o1), fmaxf(t2, o2));
        t1 = fmaxf(t1, o1);
      }
      const float g = __fadd_rn(t1, t2);
      int ahead = 0;
#pragma unroll
      for (int h = 0; h < L; ++h) {  // groups h < G (G <= L)
        const float og = __shfl_sync(kFullMask, g, seg_base + (h * gl & (L - 1)));
        ahead += h < a.G && ((og > g) || (og == g && h < grp));
      }
      if (ahead >= a.M) {
#pragma unroll
        for (int i = 0; i < 8; ++i) mine[i] = 0u;
      }
    }

    // ---- the segment's top-8 ----
    uint32_t top[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) top[i] = mine[i];
#pragma unroll
    for (int off = 1; off < L; off <<= 1) {
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = __shfl_xor_sync(kFullMask, top[i], off);
      merge8_desc(top, o);
    }

    // ---- the (K+1)-th key: in the list, or the best key below it ----
    uint32_t next;
    if (a.K < kSegTop) {
      next = pick8(top, a.K);
    } else {
      const uint32_t last = top[7];
      int taken = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) taken += mine[i] >= last;
      next = taken < 8 ? pick8(mine, taken) : 0u;
      if (taken == 8 && last != 0u) {
        // all eight of this lane's listed keys were chosen: its next key is
        // the best of the other 24, recomputed from the scores
        float b[kSegKeys];
        load_seg_row(row + e0, b);
#pragma unroll
        for (int i = 0; i < kSegKeys; ++i) b[i] = seg_score<kSoftmax>(a, b[i], smax, ssum);
        add_seg_bias(bias_j, b);
#pragma unroll
        for (int i = 0; i < kSegKeys; ++i) {
          const uint32_t k = selection_key<kKeyLow>(b[i], tag0 - (uint32_t)i);
          next = k < last ? max(next, k) : next;
        }
      }
#pragma unroll
      for (int off = 1; off < L; off <<= 1) next = max(next, __shfl_xor_sync(kFullMask, next, off));
    }

    // ---- exact unless two of the first K+1 keys agree above bit key_bits ----
    const uint32_t last = pick8(top, a.K - 1);
    bool redo = last == 0u;
#pragma unroll
    for (int r = 0; r < kSegTop; ++r) {
      if (r < a.K) {
        const uint32_t nx = r + 1 < a.K ? top[r + 1 < 8 ? r + 1 : 7] : next;
        redo = redo || ((top[r] ^ nx) >> kKeyBits) == 0u;
      }
    }

    // ---- ids (list entries j, j + L, ...) ----
    int id[kOut];
#pragma unroll
    for (int o = 0; o < kOut; ++o) id[o] = (int)(kKeyLow - (pick8(top, j + L * o) & kKeyLow));

    // ---- ties: rank the candidates by their exact keys ----
    // Let h be the high part of the (K+1)-th key, or of the K-th when the
    // two differ. Every expert of the exact top-K has a high part >= h (the
    // first K+1 keys all do, and any lower one is below all of them), and in
    // each lane those experts are a prefix of its sorted list unless the
    // whole list qualifies at a tie with the (K+1)-th key. Their exact keys
    // (order key, then expert) give each one's rank, hence its position.
    bool exact_path = redo && last == 0u;  // fewer than K candidates: the warp path decides
    if (__any_sync(kFullMask, redo && !exact_path)) {
      const bool boundary = ((last ^ next) >> kKeyBits) == 0u;
      const uint32_t h = (boundary ? next : last) >> kKeyBits;
      int c = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) c += mine[i] != 0u && (mine[i] >> kKeyBits) >= h;
      const bool over = boundary && c == 8;
      if (!redo || exact_path) c = 0;
      int incl = c;  // this lane's end offset in the segment's candidate list
#pragma unroll
      for (int off = 1; off < L; off <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, off, L);
        if (j >= off) incl += y;
      }
      const int n = __shfl_sync(kFullMask, incl, seg_base + L - 1);
      // (the ballot is taken by every lane, outside any short-circuit test)
      const unsigned over_lanes = __ballot_sync(kFullMask, over);
      const bool ok = redo && !exact_path && n <= kSegCand && (over_lanes & seg_mask) == 0u;
      if (!ok) c = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i < c) {
          const int e = (int)(kKeyLow - (mine[i] & kKeyLow));
          const float b = __fadd_rn(seg_score<kSoftmax>(a, __ldg(row + e), smax, ssum), bias_j[e - e0]);
          const uint32_t u = __float_as_uint(b);
          const uint32_t tk = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
          seg_cand[incl - c + i] = ((uint64_t)tk << 32) | (kKeyLow - (uint32_t)e);
        }
      }
      __syncwarp();
      const int c_max = __reduce_max_sync(kFullMask, c);
      for (int i = 0; i < c_max; ++i) {
        if (i < c) {
          const uint64_t x = seg_cand[incl - c + i];
          int r = 0;
          for (int m = 0; m < n; ++m) r += seg_cand[m] > x;  // keys are distinct
          if (r < a.K) seg_slot[r] = (int)(kKeyLow - (uint32_t)(x & 0xffffffffull));
        }
      }
      __syncwarp();
#pragma unroll
      for (int o = 0; o < kOut; ++o)
        if (ok && j + L * o < a.K) id[o] = seg_slot[j + L * o];
      __syncwarp();  // the candidate and slot words are reused by the next tokens
      exact_path = exact_path || (redo && !ok);
    }

    // ---- weights ----
    const bool write = live && !exact_path;
    float w[kOut];
#pragma unroll
    for (int o = 0; o < kOut; ++o) {
      const int k = j + L * o;
      w[o] = 0.0f;
      if (write && k < a.K) w[o] = seg_score<kSoftmax>(a, __ldg(row + id[o]), smax, ssum);
    }
    if (a.norm) {
      float sum = 0.0f;
#pragma unroll
      for (int k = 0; k < kSegTop; ++k)
        if (k < a.K) sum = __fadd_rn(sum, __shfl_sync(kFullMask, w[k / L], seg_base + k % L));
#pragma unroll
      for (int o = 0; o < kOut; ++o) w[o] = __fdiv_rn(w[o], sum);
    }
#pragma unroll
    for (int o = 0; o < kOut; ++o) {
      const int k = j + L * o;
      if (write && k < a.K) {
        a.ids[t * a.K + k] = id[o];
        a.weights[t * a.K + k] = __fmul_rn(w[o], a.scale);
        on_id(t, k, id[o]);
      }
    }

    // ---- tokens the ranking could not settle: the exact warp path, one at a time ----
    unsigned pending = __ballot_sync(kFullMask, live && exact_path && j == 0);
    while (pending) {
      const int l0 = __ffs(pending) - 1;
      pending &= pending - 1;
      const int64_t tr = base + l0 / L;
      route_one_token_exact<L, kSoftmax>(a, tr, warp_smem, on_id);
    }
  }
}


// Routes tokens first, first + stride, ... (below end) with the calling
// thread, all E <= EP <= 32 scores in registers. After token t's ids and
// weights are written, on_id(t, k, id) is called for k = 0 .. K-1.
template <int EP, bool kVec, typename OnId>
__device__ __forceinline__ void route_tokens_thread(const RouteArgs& a, int64_t first, int64_t end,
                                                    int64_t stride, OnId on_id) {
  float bias_r[EP];
  uint32_t valid = 0, run_start = 0, run_end = 0;
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    const bool v = e < a.E;
    bias_r[e] = v ? a.bias[e] : 0.0f;
    valid |= (uint32_t)v << e;
    if (v && e % a.S == 0) run_start |= 1u << e;
    if (v && e % a.S == a.S - 1) run_end |= 1u << e;
  }
  const bool select_groups = a.M < a.G;

  for (int64_t t = first; t < end; t += stride) {
    const float* row = a.scores + t * a.E;
    float s[EP];
    if constexpr (kVec) {
#pragma unroll
      for (int q = 0; q < EP / 4; ++q) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (4 * q < a.E) v = __ldg(reinterpret_cast<const float4*>(row + 4 * q));
        s[4 * q + 0] = v.x;
        s[4 * q + 1] = v.y;
        s[4 * q + 2] = v.z;
        s[4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < EP; ++e) s[e] = ((valid >> e) & 1u) ? __ldg(row + e) : 0.0f;
    }
    if (a.score_fn == MOE_SCORES_SOFTMAX) {
      // exp(s - max) / sum, the sum in ascending expert order
      float m = -CUDART_INF_F;
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if ((valid >> e) & 1u) m = fmaxf(m, s[e]);
      float sum = 0.0f;
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        s[e] = ((valid >> e) & 1u) ? score_exp_f32(__fsub_rn(s[e], m)) : 0.0f;
        if ((valid >> e) & 1u) sum = __fadd_rn(sum, s[e]);
      }
#pragma unroll
      for (int e = 0; e < EP; ++e) s[e] = ((valid >> e) & 1u) ? __fdiv_rn(s[e], sum) : 0.0f;
    } else if (a.score_fn != MOE_SCORES_AS_GIVEN) {
#pragma unroll
      for (int e = 0; e < EP; ++e) s[e] = apply_score_fn(a.score_fn, s[e]);
    }
    float b[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) b[e] = __fadd_rn(s[e], bias_r[e]);

    uint32_t allowed = valid;
    if (select_groups) {
      // g_end[e]: top-1 + top-2 of e's group so far; g_of[e]: the whole group's score
      float g_end[EP], g_of[EP];
      float t1 = -CUDART_INF_F, t2 = -CUDART_INF_F;
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        if ((run_start >> e) & 1u) t1 = t2 = -CUDART_INF_F;
        top2_push(t1, t2, b[e]);
        g_end[e] = (a.S == 1) ? t1 : __fadd_rn(t1, t2);
      }
      g_of[EP - 1] = g_end[EP - 1];
#pragma unroll
      for (int e = EP - 2; e >= 0; --e) g_of[e] = ((run_end >> e) & 1u) ? g_end[e] : g_of[e + 1];
      // rank each group leader against the other leaders
      uint32_t kept_leaders = 0;
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        if (!((run_start >> e) & 1u)) continue;
        int ahead = 0;
#pragma unroll
        for (int f = 0; f < EP; ++f) {
          if (!((run_start >> f) & 1u)) continue;
          ahead += (g_of[f] > g_of[e]) || (g_of[f] == g_of[e] && f < e);
        }
        if (ahead < a.M) kept_leaders |= 1u << e;
      }
      allowed = 0;
      bool keep = false;
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        if ((run_start >> e) & 1u) keep = (kept_leaders >> e) & 1u;
        if (keep && ((valid >> e) & 1u)) allowed |= 1u << e;
      }
    }

    uint32_t key[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) key[e] = ((allowed >> e) & 1u) ? ordered_key(b[e]) : 0u;

    float sum = 0.0f;
    int32_t* ids_row = a.ids + t * a.K;
    float* w_row = a.weights + t * a.K;
    for (int r = 0; r < a.K; ++r) {
      uint32_t best = 0;
      int best_e = 0;
      float best_s = 0.0f;
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (key[e] > best) { best = key[e]; best_e = e; best_s = s[e]; }
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (e == best_e) key[e] = 0u;
      ids_row[r] = best_e;
      w_row[r] = best_s;
      on_id(t, r, best_e);
      sum = __fadd_rn(sum, best_s);
    }
    for (int r = 0; r < a.K; ++r) {
      float w = w_row[r];
      if (a.norm) w = __fdiv_rn(w, sum);
      w_row[r] = __fmul_rn(w, a.scale);
    }
  }
}


inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// The shape of a router launch: which token loop runs and its template sizes.
struct RoutePlan {
  RouteArgs a;
  int C;    // warp path (E > 32): experts per lane; 0 selects the thread path
  int EP;   // thread path: E rounded up to 8, 16 or 32
  bool vec; // 16-byte score loads (E % 4 == 0 and a 16-byte aligned score matrix)
  int seg;  // segment layout: lanes per token (E = 32 * seg); 0 when it does not apply
  int staged; // staged layout: the number of groups G (E = 32 * G); 0 when it does not apply
};

// Checks the router's sizes and options and fills `p` (pointers are taken as
// given; check_route_pointers checks them).
inline moe_status_t plan_route(int32_t* expert_indices, float* expert_weights,
                        const float* expert_scores, const float* expert_bias, int64_t num_tokens,
                        int32_t n_routed_experts, int32_t n_experts_per_tok, int32_t n_groups,
                        int32_t topk_group, int32_t norm_weights, float routed_scaling_factor,
                        int32_t score_fn, RoutePlan* p) {
  const int E = n_routed_experts, K = n_experts_per_tok, G = n_groups, M = topk_group;
  if (num_tokens < 0 || E < 1 || G < 1 || M < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (E % G != 0 || M > G) return MOE_ERR_INVALID_ARG;
  const int S = E / G;
  if ((int64_t)K > (int64_t)M * S) return MOE_ERR_INVALID_ARG;
  if (E > MOE_MAX_EXPERTS || G > MOE_MAX_GROUPS || K > MOE_MAX_EXPERTS_PER_TOK)
    return MOE_ERR_UNSUPPORTED;
  if (num_tokens > (int64_t)1 << 40) return MOE_ERR_UNSUPPORTED;
  if (score_fn != MOE_SCORES_AS_GIVEN && score_fn != MOE_SCORES_SIGMOID &&
      score_fn != MOE_SCORES_SOFTMAX)
    return MOE_ERR_UNSUPPORTED;

  RouteArgs& a = p->a;
  a.ids = expert_indices;
  a.weights = expert_weights;
  a.scores = expert_scores;
  a.bias = expert_bias;
  a.T = num_tokens;
  a.E = E;
  a.K = K;
  a.G = G;
  a.M = M;
  a.S = S;
  a.norm = norm_weights != 0;
  a.scale = routed_scaling_factor;
  a.group_mode = kGroupsAllKept;
  a.seg_lanes = 1;
  a.score_fn = score_fn;
  a.warp_smem_words = 0;
  a.softmax_off = 0;
  a.key_bits = key_bits_for(E);
  a.key_low = (1u << a.key_bits) - 1u;
  p->seg = 0;
  p->staged = 0;
  p->vec = (E % 4 == 0) && aligned(expert_scores, 16);
  p->C = 0;
  p->EP = E <= 8 ? 8 : E <= 16 ? 16 : 32;
  if (E <= 32) return MOE_OK;

  p->C = E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : E <= 512 ? 16 : 32;
  if (M < G) {
    if (S % p->C == 0 && is_pow2(S / p->C)) {
      a.group_mode = kGroupsSegment;
      a.seg_lanes = S / p->C;
    } else {
      a.group_mode = kGroupsGeneric;
    }
  }
  a.softmax_off = a.group_mode == kGroupsGeneric ? E : 0;
  a.warp_smem_words = a.softmax_off + (score_fn == MOE_SCORES_SOFTMAX ? E : 0);
  // the segment layout: E a power-of-two multiple of 32, K <= 8, 16-byte
  // loads, groups of whole lanes; the warp path with C = E / 32 is its exact
  // fallback
  const int L = E / kSegKeys;
  if (E == kSegKeys * p->C && K <= kSegTop && p->vec && aligned(expert_bias, 16) &&
      (a.group_mode == kGroupsAllKept || (a.group_mode == kGroupsSegment && G <= L && L % G == 0)))
    p->seg = L;
  // the staged layout: groups of 32 experts, G = 4, 8 or 16, K <= 8, 16-byte
  // loads and bias, any score loader. The softmax loader takes it with K = 8
  // and E <= 256 (back to back at 16384 tokens, staged against segment
  // layout: 15.4 against 18.1 us for the DeepSeek-V3 shape, 10.2 against
  // 12.9 us for 128 experts all kept) except for 256 experts all kept (17.1
  // against 16.3 us), which stays on the segment layout. With every group kept
  // (topk_group == n_groups, e.g. one group) the groups play no part, so E =
  // 128 or 256 runs there as E/32 units of 32 experts, all kept (back to back
  // at 16384 tokens: 6.4 against 8.5 us for E = 128 and 9.1 against 9.9 us for
  // E = 256 on the segment layout; E = 512, 20.7 against 17.7 us, stays there).
  const int units = E / 32;
  const bool unit_shape = units * 32 == E && (units == 4 || units == 8);
  const bool softmax_ok = K == kSegTop && E <= 256 && !(M == G && E == 256);
  if (K <= kSegTop && p->vec && aligned(expert_bias, 16) &&
      (score_fn != MOE_SCORES_SOFTMAX || softmax_ok)) {
    if (S == 32 && (G == 4 || G == 8 || G == 16))
      p->staged = G;
    else if (M == G && unit_shape)
      p->staged = units;
  }
  return MOE_OK;
}

inline moe_status_t check_route_pointers(const RouteArgs& a) {
  if (!a.ids || !a.weights || !a.scores || !a.bias) return MOE_ERR_NULL_PTR;
  if (!aligned(a.ids, 4) || !aligned(a.weights, 4) || !aligned(a.scores, 4) ||
      !aligned(a.bias, 4))
    return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

// Shared memory of the warp path for `warps` warps (RouteArgs.warp_smem_words each).
inline size_t route_warp_smem(const RoutePlan& p, int warps) {
  return (size_t)warps * p.a.warp_smem_words * sizeof(float);
}

}  // namespace
}  // namespace moe
