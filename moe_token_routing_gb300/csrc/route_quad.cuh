// Quad layout of the group-limited router: four threads per token, score rows
// streamed into shared memory by bulk asynchronous copies.
//
// Page "group_limited_router_kernel", description paragraph: the experts are
// split into n_groups groups, the topk_group groups with the best scores are
// kept and n_experts_per_tok experts are chosen among them by biased score;
// Args expert_bias (selection only), expert_weights, Parameters norm_weights
// and Args routed_scaling_factor fix the weights.
//
// Shapes: groups of 32 experts, G = 4P groups (E = 128P, P = 1, 2, 4),
// K <= 8, scores as given or through the sigmoid loader, 16-byte aligned
// scores and bias.
//
// Data movement. A persistent grid of one CTA per SM splits the token rows
// into chunks of 8 rows (8*E*4 bytes, contiguous in HBM) and gives each CTA
// a contiguous run of chunks; warp w of a CTA takes chunks w, w + W, ... of
// the run. Each warp owns a ring of D chunk buffers in shared memory: lane 0
// starts D chunk copies (cp.async.bulk, completion counted by an mbarrier)
// before the warp needs the first one, and restarts a buffer with the
// warp's chunk D ahead as soon as the warp has finished with it. So up to
// W*D*8 rows per SM are in flight from the start of the kernel and the score
// loads cost no load instructions or registers.
//
// Work per token (lane 4i+q of a warp is thread q of the chunk's token i):
//  pass 1   thread q holds groups qP .. qP+P-1 and computes each one's score,
//           the fp32 sum of its two largest biased scores;
//  groups   the four threads exchange the G group scores by shuffles, rank
//           their own groups (score desc, index asc) and OR their kept bits
//           into a G-bit mask;
//  pass 2   thread q takes the kept groups number q, q+4, ... (ascending
//           group index), builds the 32-bit selection keys of their experts
//           (the order key of the biased score with the low key_bits bits
//           replaced by key_low - e, as in the segment layout) and sorts them
//           into a descending top-8 list with sorting networks of unsigned
//           min/max; two butterfly merges give all four threads the token's
//           top-8 over the kept groups.
// Only the kept groups go through the sorting networks, so a token costs
// about a third of the segment layout's instructions.
//
// Exactness: as in the segment layout, the list is the exact selection
// whenever the first K+1 keys differ above bit key_bits. Otherwise the
// candidates that can still be chosen (those whose high key part reaches
// the boundary's) are ranked by their exact 64-bit keys in shared memory,
// and a token whose candidates are not all known from the lists goes through
// the exact warp path (route_one_token_exact), which reads global memory.
//
// Waits: every wait on a chunk's mbarrier is bounded (one second). A warp
// that gives up writes expert id -1 and weight 0 for every token it has not
// routed, waits (again bounded) for its copies in flight, and returns.
#pragma once

#include "route_device.cuh"
#include "tagged_sync.cuh"

namespace moe {
namespace {

constexpr int kQuadTokens = 8;     // tokens per warp iteration (a chunk)
constexpr int kQuadCand = 16;      // tie ranking: candidate keys per token
constexpr int kQuadMaxWarps = 16;  // warps per CTA
constexpr int kQuadThreadsMax = 32 * kQuadMaxWarps;

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the asynchronous proxy (the copy
// engine that completes the transactions).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's (and, after a warp barrier, its warp's) earlier
// generic-proxy accesses of shared memory before later bulk copies into it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to this CTA's shared memory, counted on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
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

// Waits until the phase with the given parity of `bar` has completed; false
// after one second of %globaltimer or kSyncMaxPolls polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t polls = 0; polls < kSyncMaxPolls; ++polls) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kSyncTimeoutNs) return false;
  }
  return false;
}

// ------------------------------------------------------------ launch shape
// Shared memory of a quad launch with W warps and D chunk buffers per warp:
// bias [E] | mbarriers [W*D] | candidates [W*8*kQuadCand] u64 | slots
// [W*8*8] int | ring [W*D*8*E] floats (128-byte aligned).
struct QuadSmem {
  size_t bars_off, cand_off, slot_off, ring_off, total;
};

__host__ __device__ inline QuadSmem quad_smem(int E, int W, int D) {
  QuadSmem s;
  s.bars_off = ((size_t)E * sizeof(float) + 15) & ~(size_t)15;
  s.cand_off = s.bars_off + (size_t)W * D * sizeof(uint64_t);
  s.cand_off = (s.cand_off + 15) & ~(size_t)15;
  s.slot_off = s.cand_off + (size_t)W * kQuadTokens * kQuadCand * sizeof(uint64_t);
  s.ring_off = s.slot_off + (size_t)W * kQuadTokens * 8 * sizeof(int);
  s.ring_off = (s.ring_off + 127) & ~(size_t)127;
  s.total = s.ring_off + (size_t)W * D * kQuadTokens * E * sizeof(float);
  return s;
}

struct QuadShape {
  int ctas, warps, depth;
  size_t smem;
};

// One CTA per SM (fewer when there are fewer chunks). When every chunk of a
// CTA fits in flight at once (at most 16 chunks and the ring budget), each
// warp takes one chunk; otherwise 12 warps (fewer for large E) cycle through
// rings of two or more buffers.
inline QuadShape quad_shape(int64_t T, int E, int sm_count) {
  constexpr size_t kRingBudget = 192 * 1024;
  const size_t chunk_bytes = (size_t)kQuadTokens * E * sizeof(float);
  const int slots = (int)(kRingBudget / chunk_bytes);
  const int64_t chunks = (T + kQuadTokens - 1) / kQuadTokens;
  QuadShape q;
  q.ctas = (int)(chunks < sm_count ? chunks : sm_count);
  if (q.ctas < 1) q.ctas = 1;
  const int64_t per_cta = (chunks + q.ctas - 1) / q.ctas;
  const int one_shot = slots < kQuadMaxWarps ? slots : kQuadMaxWarps;
  if (per_cta <= one_shot) {
    q.warps = (int)(per_cta < 1 ? 1 : per_cta);
    q.depth = 1;
  } else {
    q.warps = slots / 2 < 12 ? slots / 2 : 12;
    q.depth = slots / q.warps;
    const int64_t per_warp = (per_cta + q.warps - 1) / q.warps;
    if (q.depth > per_warp) q.depth = (int)per_warp;
  }
  q.smem = quad_smem(E, q.warps, q.depth).total;
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
__device__ __forceinline__ uint32_t quad_key(float b, uint32_t key_low, int e) {
  const uint32_t u = __float_as_uint(b);
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return (k | key_low) - (uint32_t)e;
}

// The descending top-8 selection keys of kept group `grp` of the token whose
// staged row is `row` (32 experts, read at the rotated columns of this lane);
// all zero when `use` is false.
template <bool kSigmoid>
__device__ __forceinline__ void quad_group_top8(const RouteArgs& a, const float* row,
                                                const float* s_bias, int grp, int rot, bool use,
                                                uint32_t (&top)[8]) {
  uint32_t key[4][8];
  const float* rg = row + grp * 32;
  const float* bg = s_bias + grp * 32;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int col = ((c + rot) & 7) * 4;
    const float4 v = *reinterpret_cast<const float4*>(rg + col);
    const float4 bb = *reinterpret_cast<const float4*>(bg + col);
    const int e = grp * 32 + col;
    key[c >> 1][(c & 1) * 4 + 0] = use ? quad_key(__fadd_rn(v.x, bb.x), a.key_low, e + 0) : 0u;
    key[c >> 1][(c & 1) * 4 + 1] = use ? quad_key(__fadd_rn(v.y, bb.y), a.key_low, e + 1) : 0u;
    key[c >> 1][(c & 1) * 4 + 2] = use ? quad_key(__fadd_rn(v.z, bb.z), a.key_low, e + 2) : 0u;
    key[c >> 1][(c & 1) * 4 + 3] = use ? quad_key(__fadd_rn(v.w, bb.w), a.key_low, e + 3) : 0u;
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
__device__ __forceinline__ uint32_t quad_group_best_below(const RouteArgs& a, const float* row,
                                                          const float* s_bias, int grp,
                                                          uint32_t last) {
  uint32_t best = 0u;
  for (int i = 0; i < 32; ++i) {
    const int e = grp * 32 + i;
    const uint32_t k = quad_key(__fadd_rn(row[e], s_bias[e]), a.key_low, e);
    best = k < last ? max(best, k) : best;
  }
  return best;
}

// Routes this CTA's share of the tokens (see the top of this file); every
// thread of the CTA calls it. `smem` is the CTA's dynamic shared memory in the
// quad_smem(E, W, D) layout. After token t's ids and weights are written,
// on_id(t, k, id) is called once per k < K.
template <int P, bool kSigmoid, typename OnId>
__device__ __forceinline__ void route_tokens_quad(const RouteArgs& a, char* smem, int D,
                                                  OnId on_id) {
  constexpr int G = 4 * P;
  constexpr int E = 32 * G;
  constexpr int kRow = kQuadTokens * E;  // floats per chunk buffer
  const int W = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tq = lane >> 2;     // token of the chunk
  const int q = lane & 3;       // thread of the token
  const int rot = lane & 7;     // column rotation: a shared-memory phase's 8 lanes hit 8 bank groups
  const int qbase = lane & ~3;
  const unsigned qmask = 0xfu << qbase;

  const QuadSmem L = quad_smem(E, W, D);
  float* s_bias = reinterpret_cast<float*>(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars_off) + warp * D;
  uint64_t* tok_cand = reinterpret_cast<uint64_t*>(smem + L.cand_off) +
                       (warp * kQuadTokens + tq) * kQuadCand;
  int* tok_slot = reinterpret_cast<int*>(smem + L.slot_off) + (warp * kQuadTokens + tq) * 8;
  float* ring = reinterpret_cast<float*>(smem + L.ring_off) + (size_t)warp * D * kRow;

  const int64_t nch = (a.T + kQuadTokens - 1) / kQuadTokens;
  const int64_t c0 = nch * blockIdx.x / gridDim.x;
  const int64_t c1 = nch * (blockIdx.x + 1) / gridDim.x;
  const int64_t mine_n = c1 - c0 > warp ? (c1 - c0 - warp + W - 1) / W : 0;  // this warp's chunks

  auto issue = [&](int64_t j, int s) {
    const int64_t t0 = (c0 + warp + j * W) * kQuadTokens;
    const int64_t nt = a.T - t0 < kQuadTokens ? a.T - t0 : kQuadTokens;
    const uint32_t bytes = (uint32_t)(nt * E * sizeof(float));
    mbar_arrive_expect_tx(&bars[s], bytes);
    bulk_copy_g2s(ring + (size_t)s * kRow, a.scores + t0 * E, bytes, &bars[s]);
  };
  // the first copies start before the bias is staged
  if (lane == 0) {
    for (int s = 0; s < D; ++s) mbar_init(&bars[s], 1u);
    fence_barrier_init();
    for (int s = 0; s < D && s < mine_n; ++s) issue(s, s);
  }
  // the bias, a -0 stored as +0 (see stage_seg_bias)
  for (int i = threadIdx.x; i < E / 4; i += blockDim.x) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(a.bias) + i);
    reinterpret_cast<float4*>(s_bias)[i] = make_float4(
        __fadd_rn(v.x, 0.0f), __fadd_rn(v.y, 0.0f), __fadd_rn(v.z, 0.0f), __fadd_rn(v.w, 0.0f));
  }
  __syncthreads();

  for (int64_t j = 0; j < mine_n; ++j) {
    const int s = (int)(j % D);
    const uint32_t parity = (uint32_t)((j / D) & 1);
    const bool arrived = __all_sync(kFullMask, mbar_wait_bounded(&bars[s], parity));
    if (!arrived) {
      // give up: mark this warp's remaining tokens, then wait (bounded) for
      // the copies still in flight so that none lands after the CTA exits
      for (int64_t jj = j; jj < mine_n; ++jj) {
        const int64_t t0 = (c0 + warp + jj * W) * kQuadTokens;
        for (int i = lane; i < kQuadTokens * a.K; i += 32) {
          const int64_t t = t0 + i / a.K;
          if (t < a.T) {
            a.ids[t * a.K + i % a.K] = -1;
            a.weights[t * a.K + i % a.K] = 0.0f;
          }
        }
      }
      for (int64_t jj = j; jj < mine_n && jj < j + D; ++jj)
        mbar_wait_bounded(&bars[jj % D], (uint32_t)((jj / D) & 1));
      return;
    }

    const int64_t t = (c0 + warp + j * W) * kQuadTokens + tq;
    const bool live = t < a.T;
    float* row = ring + (size_t)s * kRow + tq * E;

    // ---- pass 1: scores of this thread's P groups ----
    float g[P];
#pragma unroll
    for (int h = 0; h < P; ++h) {
      const int grp = q * P + h;
      float* rg = row + grp * 32;
      const float* bg = s_bias + grp * 32;
      float t1 = -CUDART_INF_F, t2 = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int col = ((c + rot) & 7) * 4;
        float4 v = *reinterpret_cast<const float4*>(rg + col);
        if constexpr (kSigmoid) {
          v = make_float4(sigmoid_score(v.x), sigmoid_score(v.y), sigmoid_score(v.z),
                          sigmoid_score(v.w));
          if (live) *reinterpret_cast<float4*>(rg + col) = v;  // pass 2 and the weights read it
        }
        const float4 bb = *reinterpret_cast<const float4*>(bg + col);
        top2_push(t1, t2, __fadd_rn(v.x, bb.x));
        top2_push(t1, t2, __fadd_rn(v.y, bb.y));
        top2_push(t1, t2, __fadd_rn(v.z, bb.z));
        top2_push(t1, t2, __fadd_rn(v.w, bb.w));
      }
      g[h] = __fadd_rn(t1, t2);
    }
    if constexpr (kSigmoid) __syncwarp();

    // ---- group selection: the M best group scores, ties to the lower group ----
    uint32_t kmask = (G == 32) ? kFullMask : ((1u << G) - 1u);
    if (a.M < G) {
      float gs[G];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq)
#pragma unroll
        for (int h = 0; h < P; ++h) gs[qq * P + h] = __shfl_sync(kFullMask, g[h], qbase + qq);
      uint32_t kept = 0u;
#pragma unroll
      for (int h = 0; h < P; ++h) {
        const int x = q * P + h;
        int ahead = 0;
#pragma unroll
        for (int y = 0; y < G; ++y) ahead += (gs[y] > g[h]) || (gs[y] == g[h] && y < x);
        kept |= (uint32_t)(ahead < a.M) << x;
      }
      kept |= __shfl_xor_sync(kFullMask, kept, 1);
      kept |= __shfl_xor_sync(kFullMask, kept, 2);
      kmask = kept;
    }

    // ---- pass 2: this thread's top-8 over its kept groups, then the token's ----
    const int nkept = __popc(kmask);  // the same for every token (M, or G)
    uint32_t mine[8];
    int my_grp[P];
#pragma unroll
    for (int r = 0; r < P; ++r) {
      my_grp[r] = -1;
      if (4 * r < nkept) {
        const int idx = q + 4 * r;
        const bool use = idx < nkept;
        const int grp = use ? nth_set_bit(kmask, idx) : 0;
        my_grp[r] = use ? grp : -1;
        uint32_t lst[8];
        quad_group_top8<kSigmoid>(a, row, s_bias, grp, rot, use, lst);
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
    for (int off = 1; off < 4; off <<= 1) {
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
        // all eight of this thread's listed keys were chosen: its next key
        // is the best one below them in its kept groups
#pragma unroll
        for (int r = 0; r < P; ++r)
          if (my_grp[r] >= 0)
            next = max(next, quad_group_best_below(a, row, s_bias, my_grp[r], last));
      }
      next = max(next, __shfl_xor_sync(kFullMask, next, 1));
      next = max(next, __shfl_xor_sync(kFullMask, next, 2));
    }

    // ---- exact unless two of the first K+1 keys agree above bit key_bits ----
    const uint32_t last = pick8(top, a.K - 1);
    bool redo = last == 0u;
#pragma unroll
    for (int r = 0; r < kSegTop; ++r) {
      if (r < a.K) {
        const uint32_t nx = r + 1 < a.K ? top[r + 1 < 8 ? r + 1 : 7] : next;
        redo = redo || ((top[r] ^ nx) >> a.key_bits) == 0u;
      }
    }

    // ---- ids of this thread's outputs k = 2q, 2q+1 ----
    int id[2];
#pragma unroll
    for (int o = 0; o < 2; ++o) id[o] = (int)(a.key_low - (pick8(top, 2 * q + o) & a.key_low));

    // ---- ties: rank the candidates by their exact keys (see the segment layout) ----
    bool exact_path = redo && last == 0u;
    if (__any_sync(kFullMask, redo && !exact_path)) {
      const bool boundary = ((last ^ next) >> a.key_bits) == 0u;
      const uint32_t h = (boundary ? next : last) >> a.key_bits;
      int c = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) c += mine[i] != 0u && (mine[i] >> a.key_bits) >= h;
      const bool over = boundary && c == 8;
      if (!redo || exact_path) c = 0;
      int incl = c;  // this thread's end offset in the token's candidate list
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, off, 4);
        if (q >= off) incl += y;
      }
      const int n = __shfl_sync(kFullMask, incl, qbase + 3);
      const unsigned over_lanes = __ballot_sync(kFullMask, over);
      const bool ok = redo && !exact_path && n <= kQuadCand && (over_lanes & qmask) == 0u;
      if (!ok) c = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i < c) {
          const int e = (int)(a.key_low - (mine[i] & a.key_low));
          const float b = __fadd_rn(row[e], s_bias[e]);
          const uint32_t u = __float_as_uint(b);
          const uint32_t tk = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
          tok_cand[incl - c + i] = ((uint64_t)tk << 32) | (a.key_low - (uint32_t)e);
        }
      }
      __syncwarp();
      const int c_max = __reduce_max_sync(kFullMask, c);
      for (int i = 0; i < c_max; ++i) {
        if (i < c) {
          const uint64_t x = tok_cand[incl - c + i];
          int r = 0;
          for (int m = 0; m < n; ++m) r += tok_cand[m] > x;  // keys are distinct
          if (r < a.K) tok_slot[r] = (int)(a.key_low - (uint32_t)(x & 0xffffffffull));
        }
      }
      __syncwarp();
#pragma unroll
      for (int o = 0; o < 2; ++o)
        if (ok && 2 * q + o < a.K) id[o] = tok_slot[2 * q + o];
      __syncwarp();  // the candidate and slot words are reused by the next chunk
      exact_path = exact_path || (redo && !ok);
    }

    // ---- weights: unbiased score, optional normalisation, scaling ----
    const bool write = live && !exact_path;
    float w[2];
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      const int k = 2 * q + o;
      w[o] = (write && k < a.K) ? row[id[o]] : 0.0f;
    }
    if (a.norm) {
      float sum = 0.0f;
#pragma unroll
      for (int k = 0; k < kSegTop; ++k)
        if (k < a.K) sum = __fadd_rn(sum, __shfl_sync(kFullMask, w[k & 1], qbase + (k >> 1)));
#pragma unroll
      for (int o = 0; o < 2; ++o) w[o] = __fdiv_rn(w[o], sum);
    }
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      const int k = 2 * q + o;
      if (write && k < a.K) {
        a.ids[t * a.K + k] = id[o];
        a.weights[t * a.K + k] = __fmul_rn(w[o], a.scale);
        on_id(t, k, id[o]);
      }
    }

    // ---- tokens the ranking could not settle: the exact warp path, one at a time ----
    unsigned pending = __ballot_sync(kFullMask, live && exact_path && q == 0);
    while (pending) {
      const int l0 = __ffs(pending) - 1;
      pending &= pending - 1;
      route_one_token_exact<E / 32, false>(a, t - tq + (l0 >> 2), nullptr, on_id);
    }

    // ---- the buffer is free: start the copy of this warp's chunk D ahead ----
    __syncwarp();
    if (lane == 0 && j + D < mine_n) {
      fence_proxy_async_smem();
      issue(j + D, s);
    }
  }
}

// Launches a quad-layout kernel (arguments: `args`, then the ring depth) in
// the shape quad_shape picks for T tokens and E experts.
template <typename Args>
moe_status_t launch_quad(void (*kernel)(Args, int), const Args& args, int64_t T, int E,
                         cudaStream_t stream) {
  const QuadShape q = quad_shape(T, E, device_info().sm_count);
  if (q.smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)q.smem) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return launch(kernel, q.ctas, 32 * q.warps, q.smem, stream, args, q.depth);
}

}  // namespace
}  // namespace moe
