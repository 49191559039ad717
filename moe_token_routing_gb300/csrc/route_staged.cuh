// Staged layout of the group-limited router: R threads per token (R = 2 or
// 4), score rows streamed into shared memory by bulk asynchronous copies.
//
// Page "group_limited_router_kernel", description paragraph: the experts are
// split into n_groups groups, the topk_group groups with the best scores are
// kept and n_experts_per_tok experts are chosen among them by biased score;
// Args expert_bias (selection only), expert_weights, Parameters norm_weights
// and Args routed_scaling_factor fix the weights.
//
// Shapes: groups of 32 experts, G = R*P groups (P groups per thread in the
// first pass), K <= 8, scores as given or through the sigmoid loader, 16-byte
// aligned scores and bias. With every group kept (topk_group == n_groups)
// the group size does not matter and G counts units of 32 experts.
//
// Data movement. A persistent grid of one CTA per SM splits the token rows
// into chunks of 32/R rows (contiguous in HBM) and gives each CTA a
// contiguous run of chunks; warp w of a CTA takes chunks w, w + W, ... of the
// run. Each warp owns a ring of D chunk buffers in shared memory: lane 0
// starts D chunk copies (cp.async.bulk, completion counted by an mbarrier)
// before the warp needs the first one, and restarts a buffer with the
// warp's chunk D ahead as soon as the warp has finished with it. Up to W*D
// chunks per SM are in flight from the start of the kernel, and the score
// loads cost no load instructions or registers.
//
// Work per token (lane R*i + h of a warp is thread h of the chunk's token i):
//  pass 1   thread h holds groups hP .. hP+P-1; the fp32 sum of each group's
//           two largest biased scores is its score;
//  groups   the R threads exchange the group scores' order keys and rank
//           their own groups (score desc, index asc); OR-ing the kept bits
//           over the R threads gives a G-bit mask;
//  pass 2   thread h takes the kept groups number h, h+R, ... (ascending
//           group index), builds the 32-bit selection keys of their experts
//           (the order key of the biased score with the low key_bits bits
//           replaced by key_low - e) and sorts them into a descending top-8
//           list with sorting networks of unsigned min/max; log2(R) butterfly
//           merges give every thread of the token the token's top-8.
// Only the kept groups go through the sorting networks. When the smallest
// second-best score of the kept groups is >= 0 for every token of the warp,
// every expert that can be chosen has a non-negative biased score, and the
// key is one logic operation: the high bits of the float with its sign bit
// flipped. A negative score then gets a key below every non-negative one,
// which is all the selection needs of it.
//
// Exactness: the list is the exact selection whenever the first K+1 keys
// differ above bit key_bits. Otherwise the candidates that can still be
// chosen (those whose high key part reaches the boundary's) are ranked by
// their exact 64-bit keys in shared memory, and a token whose candidates are
// not all known from the lists goes through the exact warp path
// (route_one_token_exact), which reads global memory.
//
// Waits: every wait on a chunk's mbarrier is bounded (one second). A warp
// that gives up writes expert id -1 and weight 0 for every token it has not
// routed, waits (again bounded) for its copies in flight, and returns.
#pragma once

#include "mbarrier.cuh"
#include "route_device.cuh"

namespace moe {
namespace {

constexpr int kStagedR = 4;          // threads per token of the product kernels
constexpr int kStagedCand = 16;      // tie ranking: candidate keys per token
constexpr int kStagedMaxWarps = 16;  // warps per CTA
constexpr int kStagedThreadsMax = 32 * kStagedMaxWarps;

// max(a, b, c) in one instruction (three-operand max.f32, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ------------------------------------------------------------ launch shape
// Shared memory of a staged launch with W warps and D chunk buffers per warp:
// bias [E] | mbarriers [W*D] | candidates [W*tokens*kStagedCand] u64 | slots
// [W*tokens*8] int | ring [W*D*tokens*E] floats (128-byte aligned), with
// `tokens` = 32/R tokens per chunk.
struct StagedSmem {
  size_t bars_off, cand_off, slot_off, ring_off, total;
};

__host__ __device__ inline StagedSmem staged_smem(int E, int tokens, int W, int D) {
  StagedSmem s;
  s.bars_off = ((size_t)E * sizeof(float) + 15) & ~(size_t)15;
  s.cand_off = s.bars_off + (size_t)W * D * sizeof(uint64_t);
  s.cand_off = (s.cand_off + 15) & ~(size_t)15;
  s.slot_off = s.cand_off + (size_t)W * tokens * kStagedCand * sizeof(uint64_t);
  s.ring_off = s.slot_off + (size_t)W * tokens * 8 * sizeof(int);
  s.ring_off = (s.ring_off + 127) & ~(size_t)127;
  s.total = s.ring_off + (size_t)W * D * tokens * E * sizeof(float);
  return s;
}

struct StagedShape {
  int ctas, warps, depth;
  size_t smem;
};

// What a staged kernel needs of its shape: the ring depth and the split of
// the chunks over the CTAs (CTA b takes per_cta chunks, one more if b < rem).
struct StagedSplit {
  int depth;
  int rem;
  int64_t per_cta;
};

// One CTA per SM (fewer when there are fewer chunks). When every chunk of a
// CTA fits in flight at once (at most 16 chunks and the ring budget), each
// warp takes one chunk; otherwise the CTA's warps cycle through rings of two
// or more buffers, as many warps as the ring budget allows with two each (at
// most 12).
inline StagedShape staged_shape(int64_t T, int E, int tokens, int sm_count) {
  constexpr size_t kRingBudget = 192 * 1024;
  const size_t chunk_bytes = (size_t)tokens * E * sizeof(float);
  const int slots = (int)(kRingBudget / chunk_bytes);
  const int64_t chunks = (T + tokens - 1) / tokens;
  StagedShape q;
  q.ctas = (int)(chunks < sm_count ? chunks : sm_count);
  if (q.ctas < 1) q.ctas = 1;
  const int64_t per_cta = (chunks + q.ctas - 1) / q.ctas;
  const int one_shot = slots < kStagedMaxWarps ? slots : kStagedMaxWarps;
  if (per_cta <= one_shot) {
    q.warps = (int)(per_cta < 1 ? 1 : per_cta);
    q.depth = 1;
  } else {
    q.warps = slots / 2 < 12 ? slots / 2 : 12;
    q.depth = slots / q.warps;
    const int64_t per_warp = (per_cta + q.warps - 1) / q.warps;
    if (q.depth > per_warp) q.depth = (int)per_warp;
  }
  q.smem = staged_smem(E, tokens, q.warps, q.depth).total;
  return q;
}

// ------------------------------------------------------------ token loop
// Index of the n-th (from 0) set bit of m (m has more than n set bits).
__device__ __forceinline__ int nth_set_bit(uint32_t m, int n) {
  for (int i = 0; i < n; ++i) m &= m - 1u;
  return __ffs(m) - 1;
}

__device__ __forceinline__ float sigmoid_score(float x) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, score_exp_f32(-x)));
}

// Selection key of expert e from its biased score b (b is never -0: the
// staged bias holds no -0).
__device__ __forceinline__ uint32_t staged_key(float b, uint32_t key_low, int e) {
  const uint32_t u = __float_as_uint(b);
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return (k | key_low) - (uint32_t)e;
}

// The same key for b >= 0 from `tag` = 0x80000000 | (key_low - e): the high
// bits of b with the sign bit flipped, then the tag. For b < 0 it gives a key
// below 0x80000000, so below every b >= 0.
__device__ __forceinline__ uint32_t staged_key_nonneg(float b, uint32_t key_low, uint32_t tag) {
  return (__float_as_uint(b) & ~key_low) ^ tag;
}

// The descending top-8 selection keys of kept group `grp` of the token whose
// staged row is `row` (32 experts, read at the rotated columns of this lane).
template <bool kNonneg, uint32_t kKeyLow>
__device__ __forceinline__ void staged_group_top8(const float* row, const float* s_bias, int grp,
                                                  int rot, uint32_t (&top)[8]) {
  uint32_t key[4][8];
  const float* rg = row + grp * 32;
  const float* bg = s_bias + grp * 32;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int col = ((c + rot) & 7) * 4;
    const float4 v = *reinterpret_cast<const float4*>(rg + col);
    const float4 bb = *reinterpret_cast<const float4*>(bg + col);
    const int e = grp * 32 + col;
    const float b0 = __fadd_rn(v.x, bb.x), b1 = __fadd_rn(v.y, bb.y);
    const float b2 = __fadd_rn(v.z, bb.z), b3 = __fadd_rn(v.w, bb.w);
    uint32_t* k = &key[c >> 1][(c & 1) * 4];
    if constexpr (kNonneg) {
      const uint32_t tag = 0x80000000u | (kKeyLow - (uint32_t)e);
      k[0] = staged_key_nonneg(b0, kKeyLow, tag);
      k[1] = staged_key_nonneg(b1, kKeyLow, tag - 1u);
      k[2] = staged_key_nonneg(b2, kKeyLow, tag - 2u);
      k[3] = staged_key_nonneg(b3, kKeyLow, tag - 3u);
    } else {
      k[0] = staged_key(b0, kKeyLow, e + 0);
      k[1] = staged_key(b1, kKeyLow, e + 1);
      k[2] = staged_key(b2, kKeyLow, e + 2);
      k[3] = staged_key(b3, kKeyLow, e + 3);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) sort8_desc(key[i]);
  merge8_desc(key[0], key[1]);
  merge8_desc(key[2], key[3]);
  merge8_desc(key[0], key[2]);
#pragma unroll
  for (int i = 0; i < 8; ++i) top[i] = key[0][i];
}

// Best key below `last` in kept group `grp` (0 if none).
template <uint32_t kKeyLow>
__device__ __forceinline__ uint32_t staged_group_best_below(const float* row, const float* s_bias,
                                                            int grp, uint32_t last) {
  uint32_t best = 0u;
  for (int i = 0; i < 32; ++i) {
    const int e = grp * 32 + i;
    const uint32_t k = staged_key(__fadd_rn(row[e], s_bias[e]), kKeyLow, e);
    best = k < last ? max(best, k) : best;
  }
  return best;
}

// top[h*kOut + o] for thread h of R (kOut = 8/R entries each), by selects
// on the bits of h instead of a run-time index.
template <int R, int kOut>
__device__ __forceinline__ uint32_t pick_for_thread(const uint32_t (&top)[8], int h, int o) {
  if constexpr (R == 2) {
    return (h & 1) ? top[4 + o] : top[o];
  } else {
    const uint32_t lo = (h & 1) ? top[2 + o] : top[o];
    const uint32_t hi = (h & 1) ? top[6 + o] : top[4 + o];
    return (h & 2) ? hi : lo;
  }
}

// Order key of an fp32 value (see ordered_key), unsigned: a > b iff key(a) >
// key(b); +0 and -0 share a key; never 0 for a non-NaN value.
__device__ __forceinline__ uint32_t score_order_key(float v) { return ordered_key(v); }

// Routes this CTA's share of the tokens (see the top of this file); every
// thread of the CTA calls it. `smem` is the CTA's dynamic shared memory in the
// staged_smem(E, 32/R, W, D) layout. After token t's ids and weights are
// written, on_id(t, k, id) is called once per k < K.
template <int R, int P, bool kSigmoid, int kKc, bool kSoftmax, typename OnId>
__device__ __forceinline__ void route_tokens_staged(const RouteArgs& a, char* smem,
                                                    const StagedSplit& sp, OnId on_id) {
  const int D = sp.depth;
  static_assert(R == 2 || R == 4, "two or four threads per token");
  static_assert(!(kSigmoid && kSoftmax), "one score loader");
  static_assert(kKc >= 0 && kKc <= kSegTop, "K fixed at compile time (1 .. 8) or 0");
  const int K = kKc > 0 ? kKc : a.K;  // experts per token
  constexpr int G = R * P;
  constexpr int E = 32 * G;
  constexpr int kTok = 32 / R;           // tokens per chunk
  constexpr int kOut = kSegTop / R;      // list entries (picks) per thread
  constexpr int kRow = kTok * E;         // floats per chunk buffer
  constexpr int kKeyBits = key_bits_for(E);  // equal to a.key_bits (the same function)
  constexpr uint32_t kKeyLow = (1u << kKeyBits) - 1u;
  const int W = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tq = lane / R;       // token of the chunk
  const int h = lane % R;        // thread of the token
  const int rot = lane & 7;      // column rotation: a shared-memory phase's 8 lanes hit 8 bank groups
  const int tbase = lane & ~(R - 1);
  const unsigned tmask = ((1u << R) - 1u) << tbase;

  const StagedSmem L = staged_smem(E, kTok, W, D);
  float* s_bias = reinterpret_cast<float*>(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars_off) + warp * D;
  uint64_t* tok_cand = reinterpret_cast<uint64_t*>(smem + L.cand_off) +
                       (warp * kTok + tq) * kStagedCand;
  int* tok_slot = reinterpret_cast<int*>(smem + L.slot_off) + (warp * kTok + tq) * 8;
  float* ring = reinterpret_cast<float*>(smem + L.ring_off) + (size_t)warp * D * kRow;

  // a thread's kOut picks are consecutive in a 32-byte row when K = 8: one
  // vector store each for ids and weights if the rows are aligned
  const bool vec_out = K == kSegTop &&
                       ((reinterpret_cast<uintptr_t>(a.ids) | reinterpret_cast<uintptr_t>(a.weights)) &
                        (sizeof(int32_t) * kOut - 1)) == 0;
  // this CTA's chunks [c0, c1): an even split (the host passes nch / ctas and
  // nch % ctas, so no division runs here); this warp's are c0 + warp, + W, ...
  const int64_t c0 = (int64_t)blockIdx.x * sp.per_cta +
                     ((int)blockIdx.x < sp.rem ? (int)blockIdx.x : sp.rem);
  const int64_t c1 = c0 + sp.per_cta + ((int)blockIdx.x < sp.rem ? 1 : 0);
  const int64_t ahead = (int64_t)D * W;  // chunks between a buffer's two uses

  auto issue = [&](int64_t ch, int s) {
    const int64_t t0 = ch * kTok;
    const int64_t nt = a.T - t0 < kTok ? a.T - t0 : kTok;
    const uint32_t bytes = (uint32_t)(nt * E * sizeof(float));
    mbar_arrive_expect_tx(&bars[s], bytes);
    bulk_copy_g2s(ring + (size_t)s * kRow, a.scores + t0 * E, bytes, &bars[s]);
  };
  // The bias loads go out first (a load issued after the chunk copies waits
  // behind them at the memory), then lane 0 of each warp starts its first D
  // chunk copies; the bias reaches shared memory while they are in flight.
  constexpr int kBiasPer = (E / 4 + 31) / 32;  // float4 loads per thread at W = 1
  float4 bv[kBiasPer];
#pragma unroll
  for (int q = 0; q < kBiasPer; ++q) {
    const int i = threadIdx.x + q * blockDim.x;
    if (i < E / 4) bv[q] = __ldg(reinterpret_cast<const float4*>(a.bias) + i);
  }
  if (lane == 0) {
    for (int s = 0; s < D; ++s) mbar_init(&bars[s], 1u);
    fence_barrier_init();
    for (int s = 0; s < D && c0 + warp + (int64_t)s * W < c1; ++s) issue(c0 + warp + (int64_t)s * W, s);
  }
  // the bias, a -0 stored as +0 (see stage_seg_bias)
#pragma unroll
  for (int q = 0; q < kBiasPer; ++q) {
    const int i = threadIdx.x + q * blockDim.x;
    if (i < E / 4)
      reinterpret_cast<float4*>(s_bias)[i] =
          make_float4(__fadd_rn(bv[q].x, 0.0f), __fadd_rn(bv[q].y, 0.0f), __fadd_rn(bv[q].z, 0.0f),
                      __fadd_rn(bv[q].w, 0.0f));
  }
  __syncthreads();

  int s = 0;            // ring buffer of this warp's j-th chunk (j mod D)
  uint32_t parity = 0;  // its mbarrier phase parity ((j / D) mod 2)
  for (int64_t ch = c0 + warp; ch < c1;
       ch += W, s = s + 1 < D ? s + 1 : 0, parity ^= s == 0 ? 1u : 0u) {
    const bool arrived = __all_sync(kFullMask, mbar_wait_bounded(&bars[s], parity));
    if (!arrived) {
      // give up: mark this warp's remaining tokens, then wait (bounded) for
      // the copies still in flight so that none lands after the CTA exits
      for (int64_t cc = ch; cc < c1; cc += W) {
        for (int i = lane; i < kTok * K; i += 32) {
          const int64_t t = cc * kTok + i / K;
          if (t < a.T) {
            a.ids[t * K + i % K] = -1;
            a.weights[t * K + i % K] = 0.0f;
          }
        }
      }
      int ss = s;
      uint32_t pp = parity;
      for (int64_t cc = ch; cc < c1 && cc < ch + ahead; cc += W) {
        mbar_wait_bounded(&bars[ss], pp);
        if (++ss == D) {
          ss = 0;
          pp ^= 1u;
        }
      }
      return;
    }

    const int64_t t = ch * kTok + tq;
    const bool live = t < a.T;
    float* row = ring + (size_t)s * kRow + tq * E;

    // ---- softmax loader: the row's max, exp(x - max) over the row, and the
    // fp32 sum of those in ascending expert order (thread h's experts follow
    // those of threads 0 .. h-1, so the running sum passes from thread to
    // thread); pass 1 divides by it ----
    float ssum = 1.0f;
    if constexpr (kSoftmax) {
      float m = -CUDART_INF_F;
#pragma unroll
      for (int i = 0; i < P; ++i) {
        const float* rg = row + (h * P + i) * 32;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 v = *reinterpret_cast<const float4*>(rg + ((c + rot) & 7) * 4);
          m = fmaxf(fmaxf(m, fmaxf(v.x, v.y)), fmaxf(v.z, v.w));
        }
      }
#pragma unroll
      for (int off = 1; off < R; off <<= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, off));
#pragma unroll
      for (int i = 0; i < P; ++i) {
        float* rg = row + (h * P + i) * 32;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float4* q = reinterpret_cast<float4*>(rg + ((c + rot) & 7) * 4);
          const float4 v = *q;
          const float4 e = make_float4(score_exp_f32(__fsub_rn(v.x, m)), score_exp_f32(__fsub_rn(v.y, m)),
                                       score_exp_f32(__fsub_rn(v.z, m)), score_exp_f32(__fsub_rn(v.w, m)));
          if (live) *q = e;
        }
      }
      float run = 0.0f;
#pragma unroll
      for (int l = 0; l < R; ++l) {
        if (h == l) {
#pragma unroll
          for (int i = 0; i < P; ++i) {
            const float* rg = row + (h * P + i) * 32;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const float4 e = *reinterpret_cast<const float4*>(rg + c * 4);
              run = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(run, e.x), e.y), e.z), e.w);
            }
          }
        }
        run = __shfl_sync(kFullMask, run, tbase + l);
      }
      ssum = run;
    }

    // ---- pass 1: scores of this thread's P groups (top-2 of each float4 by
    // two min/max pairs, then the eight float4 top-2s merged as a tree, so the
    // merges of a group form three dependent levels rather than a chain) ----
    uint32_t gk[P];   // order keys of the group scores
    float sec[P];     // second-best biased score of each group
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const int grp = h * P + i;
      float* rg = row + grp * 32;
      const float* bg = s_bias + grp * 32;
      float q1[8], q2[8];  // top-2 of each float4
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int col = ((c + rot) & 7) * 4;
        float4 v = *reinterpret_cast<const float4*>(rg + col);
        if constexpr (kSigmoid) {
          v = make_float4(sigmoid_score(v.x), sigmoid_score(v.y), sigmoid_score(v.z),
                          sigmoid_score(v.w));
          if (live) *reinterpret_cast<float4*>(rg + col) = v;  // pass 2 and the weights read it
        }
        if constexpr (kSoftmax) {
          v = make_float4(__fdiv_rn(v.x, ssum), __fdiv_rn(v.y, ssum), __fdiv_rn(v.z, ssum),
                          __fdiv_rn(v.w, ssum));
          if (live) *reinterpret_cast<float4*>(rg + col) = v;  // pass 2 and the weights read it
        }
        const float4 bb = *reinterpret_cast<const float4*>(bg + col);
        const float x = __fadd_rn(v.x, bb.x), y = __fadd_rn(v.y, bb.y);
        const float z = __fadd_rn(v.z, bb.z), w = __fadd_rn(v.w, bb.w);
        const float hi1 = fmaxf(x, y), lo1 = fminf(x, y);
        const float hi2 = fmaxf(z, w), lo2 = fminf(z, w);
        q1[c] = fmaxf(hi1, hi2);
        q2[c] = fmax3(fminf(hi1, hi2), lo1, lo2);
      }
      // merge (a1, a2) with (b1, b2): the larger first, and the larger of the
      // smaller first and both seconds
#pragma unroll
      for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int c = 0; c < w; ++c) {
          q2[c] = fmax3(fminf(q1[c], q1[c + w]), q2[c], q2[c + w]);
          q1[c] = fmaxf(q1[c], q1[c + w]);
        }
      gk[i] = score_order_key(__fadd_rn(q1[0], q2[0]));
      sec[i] = q2[0];
    }
    if constexpr (kSigmoid || kSoftmax) __syncwarp();

    // ---- group selection: the M best group scores, ties to the lower group ----
    uint32_t kmask = (G == 32) ? kFullMask : ((1u << G) - 1u);
    // (with every group kept, G counts units of 32 experts, all kept)
    if (a.group_mode != kGroupsAllKept && a.M < G) {
      // ahead[i]: groups that beat own group x = hP + i. The other threads'
      // groups are visited by distance d = 1 .. R-1 (thread (h + d) mod R);
      // those of a thread before h have lower indices, so they beat x on an
      // equal key too (key >= gk, i.e. key > gk - 1; group keys are >= 1).
      int ahead[P];
#pragma unroll
      for (int i = 0; i < P; ++i) {
        ahead[i] = 0;
#pragma unroll
        for (int l = 0; l < P; ++l)
          if (l != i) ahead[i] += l < i ? (gk[l] >= gk[i]) : (gk[l] > gk[i]);
      }
#pragma unroll
      for (int d = 1; d < R; ++d) {
        const int src = tbase + ((h + d) & (R - 1));
        const bool lower = h + d >= R;  // that thread's groups precede ours
        uint32_t o[P];
#pragma unroll
        for (int l = 0; l < P; ++l) o[l] = __shfl_sync(kFullMask, gk[l], src);
#pragma unroll
        for (int i = 0; i < P; ++i) {
          const uint32_t thr = gk[i] - (lower ? 1u : 0u);
#pragma unroll
          for (int l = 0; l < P; ++l) ahead[i] += o[l] > thr;
        }
      }
      uint32_t kept = 0u;
#pragma unroll
      for (int i = 0; i < P; ++i) kept |= (uint32_t)(ahead[i] < a.M) << i;
      kept <<= h * P;
#pragma unroll
      for (int off = 1; off < R; off <<= 1) kept |= __shfl_xor_sync(kFullMask, kept, off);
      kmask = kept;
    }

    // ---- threshold: the smallest second-best score of the kept groups; every
    // expert the token can choose has a biased score >= it ----
    float tau = CUDART_INF_F;
#pragma unroll
    for (int i = 0; i < P; ++i)
      if ((kmask >> (h * P + i)) & 1u) tau = fminf(tau, sec[i]);
#pragma unroll
    for (int off = 1; off < R; off <<= 1) tau = fminf(tau, __shfl_xor_sync(kFullMask, tau, off));
    // (each kept group has two scores >= tau, so with 2*nkept >= K every
    // chosen expert has one too)
    const int nkept = __popc(kmask);  // M (or G), the same for every token
    const bool nonneg = __all_sync(kFullMask, 2 * nkept >= K && (!live || tau >= 0.0f));

    // ---- pass 2: this thread's top-8 over its kept groups, then the token's ----
    uint32_t mine[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mine[i] = 0u;
    int my_grp[P];
#pragma unroll
    for (int r = 0; r < P; ++r) {
      my_grp[r] = -1;
      if (R * r < nkept) {
        const int idx = h + R * r;
        const bool use = idx < nkept;
        const int grp = use ? nth_set_bit(kmask, idx) : 0;
        my_grp[r] = use ? grp : -1;
        uint32_t lst[8];
        if (nonneg)
          staged_group_top8<true, kKeyLow>(row, s_bias, grp, rot, lst);
        else
          staged_group_top8<false, kKeyLow>(row, s_bias, grp, rot, lst);
#pragma unroll
        for (int i = 0; i < 8; ++i) lst[i] = use ? lst[i] : 0u;
        if (r == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) mine[i] = lst[i];
        } else {
          merge8_desc(mine, lst);
        }
      }
    }
    uint32_t top[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) top[i] = mine[i];
#pragma unroll
    for (int off = 1; off < R; off <<= 1) {
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = __shfl_xor_sync(kFullMask, top[i], off);
      merge8_desc(top, o);
    }

    // ---- the (K+1)-th key: in the list, or the best key below it ----
    uint32_t next;
    if (K < kSegTop) {
      next = pick8(top, K);
    } else {
      const uint32_t last = top[7];
      int taken = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) taken += mine[i] >= last;
      next = taken < 8 ? pick8(mine, taken) : 0u;
      if (taken == 8 && last != 0u) {
        // all eight of this thread's listed keys were chosen: its next key
        // is the best one below them in its kept groups
#pragma unroll
        for (int r = 0; r < P; ++r)
          if (my_grp[r] >= 0)
            next = max(next, staged_group_best_below<kKeyLow>(row, s_bias, my_grp[r], last));
      }
#pragma unroll
      for (int off = 1; off < R; off <<= 1)
        next = max(next, __shfl_xor_sync(kFullMask, next, off));
    }

    // ---- exact unless two of the first K+1 keys agree above bit key_bits ----
    const uint32_t last = pick8(top, K - 1);
    bool redo = last == 0u;
#pragma unroll
    for (int r = 0; r < kSegTop; ++r) {
      if (r < K) {
        const uint32_t nx = r + 1 < K ? top[r + 1 < 8 ? r + 1 : 7] : next;
        redo = redo || ((top[r] ^ nx) >> kKeyBits) == 0u;
      }
    }

    // ---- ids of this thread's picks k = h*kOut + o ----
    int id[kOut];
#pragma unroll
    for (int o = 0; o < kOut; ++o)
      id[o] = (int)(kKeyLow - (pick_for_thread<R, kOut>(top, h, o) & kKeyLow));

    // ---- ties: rank the candidates by their exact keys (see the segment layout) ----
    bool exact_path = redo && last == 0u;
    if (__any_sync(kFullMask, redo && !exact_path)) {
      const bool boundary = ((last ^ next) >> kKeyBits) == 0u;
      const uint32_t hk = (boundary ? next : last) >> kKeyBits;
      int c = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) c += mine[i] != 0u && (mine[i] >> kKeyBits) >= hk;
      const bool over = boundary && c == 8;
      if (!redo || exact_path) c = 0;
      int incl = c;  // this thread's end offset in the token's candidate list
#pragma unroll
      for (int off = 1; off < R; off <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, off, R);
        if (h >= off) incl += y;
      }
      const int n = __shfl_sync(kFullMask, incl, tbase + R - 1);
      const unsigned over_lanes = __ballot_sync(kFullMask, over);
      const bool ok = redo && !exact_path && n <= kStagedCand && (over_lanes & tmask) == 0u;
      if (!ok) c = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i < c) {
          const int e = (int)(kKeyLow - (mine[i] & kKeyLow));
          const float b = __fadd_rn(row[e], s_bias[e]);
          const uint32_t u = __float_as_uint(b);
          const uint32_t tk = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
          tok_cand[incl - c + i] = ((uint64_t)tk << 32) | (kKeyLow - (uint32_t)e);
        }
      }
      __syncwarp();
      const int c_max = __reduce_max_sync(kFullMask, c);
      for (int i = 0; i < c_max; ++i) {
        if (i < c) {
          const uint64_t x = tok_cand[incl - c + i];
          int r = 0;
          for (int m = 0; m < n; ++m) r += tok_cand[m] > x;  // keys are distinct
          if (r < K) tok_slot[r] = (int)(kKeyLow - (uint32_t)(x & 0xffffffffull));
        }
      }
      __syncwarp();
#pragma unroll
      for (int o = 0; o < kOut; ++o)
        if (ok && h * kOut + o < K) id[o] = tok_slot[h * kOut + o];
      __syncwarp();  // the candidate and slot words are reused by the next chunk
      exact_path = exact_path || (redo && !ok);
    }

    // ---- weights: unbiased score, optional normalisation, scaling ----
    const bool write = live && !exact_path;
    float w[kOut];
#pragma unroll
    for (int o = 0; o < kOut; ++o) {
      const int k = h * kOut + o;
      w[o] = (write && k < K) ? row[id[o]] : 0.0f;
    }
    if (a.norm) {
      float sum = 0.0f;
#pragma unroll
      for (int k = 0; k < kSegTop; ++k)
        if (k < K)
          sum = __fadd_rn(sum, __shfl_sync(kFullMask, w[k % kOut], tbase + k / kOut));
#pragma unroll
      for (int o = 0; o < kOut; ++o) w[o] = __fdiv_rn(w[o], sum);
    }
#pragma unroll
    for (int o = 0; o < kOut; ++o) w[o] = __fmul_rn(w[o], a.scale);
    if (write) {
      if (vec_out) {
        int32_t* ip = a.ids + t * kSegTop + h * kOut;
        float* wp = a.weights + t * kSegTop + h * kOut;
        if constexpr (kOut == 4) {
          *reinterpret_cast<int4*>(ip) = make_int4(id[0], id[1], id[2], id[3]);
          *reinterpret_cast<float4*>(wp) = make_float4(w[0], w[1], w[2], w[3]);
        } else {
          *reinterpret_cast<int2*>(ip) = make_int2(id[0], id[1]);
          *reinterpret_cast<float2*>(wp) = make_float2(w[0], w[1]);
        }
      } else {
#pragma unroll
        for (int o = 0; o < kOut; ++o) {
          const int k = h * kOut + o;
          if (k < K) {
            a.ids[t * K + k] = id[o];
            a.weights[t * K + k] = w[o];
          }
        }
      }
#pragma unroll
      for (int o = 0; o < kOut; ++o)
        if (h * kOut + o < K) on_id(t, h * kOut + o, id[o]);
    }

    // ---- tokens the ranking could not settle: the exact warp path, one at a time ----
    unsigned pending = __ballot_sync(kFullMask, live && exact_path && h == 0);
    while (pending) {
      const int l0 = __ffs(pending) - 1;
      pending &= pending - 1;
      // (the softmax loader's strip: this warp's ring buffer, whose chunk is done)
      route_one_token_exact<E / 32, kSoftmax>(a, t - tq + l0 / R,
                                              kSoftmax ? ring + (size_t)s * kRow : nullptr, on_id);
    }

    // ---- the buffer is free: start the copy of this warp's chunk D ahead ----
    __syncwarp();
    if (lane == 0 && ch + ahead < c1) {
      fence_proxy_async_smem();
      issue(ch + ahead, s);
    }
  }
}

// Launches a staged-layout kernel (arguments: `args`, then its StagedSplit)
// with `tokens` tokens per chunk, in the shape staged_shape picks for T
// tokens and E experts.
template <typename Args>
moe_status_t launch_staged(void (*kernel)(Args, StagedSplit), const Args& args, int64_t T, int E,
                           int tokens, cudaStream_t stream) {
  const StagedShape q = staged_shape(T, E, tokens, device_info().sm_count);
  if (q.smem > 48 * 1024 && set_dynamic_smem((const void*)kernel, q.smem) != MOE_OK)
    return MOE_ERR_CUDA;
  const int64_t chunks = (T + tokens - 1) / tokens;
  StagedSplit sp;
  sp.depth = q.depth;
  sp.per_cta = chunks / q.ctas;
  sp.rem = (int)(chunks % q.ctas);
  return launch(kernel, q.ctas, 32 * q.warps, q.smem, stream, args, sp);
}

}  // namespace
}  // namespace moe
