// Router + expert index builder for sm_103a: what moe_route followed by
// moe_create_indices computes, in two designs.
//
// Page "group_limited_router_kernel" fixes the routing (description
// paragraph; Args expert_indices, expert_weights); page "moe_create_indices"
// fixes the stable bucket sort by expert, the compact CSR, the inverse
// permutation and the usage stats (description paragraph; Args
// token_expert_order .. expert_usage_stats, scales_offset_p).
//
// moe_route_index (three launches, at the end of this file): the router adds
// each slot it writes to counts[expert][slot / 1024], and the index builder's
// row-prefix and scatter kernels (index_device.cuh) follow, so the separate
// count kernel and its re-read of the ids disappear.
//
// moe_route_index_single_launch (one cooperative launch, described here):
// CTA b owns a contiguous range of tokens and each of its warps a contiguous
// part of that range, so the slots t*K+k of a warp form one contiguous slot
// range and a stable placement needs only per-warp counts:
//   phase 1  each warp routes its tokens with the router's own token loops
//            and counts the chosen experts in shared memory; the CTA
//            publishes its count of each expert e as cnt[e][b].
//   phase 2  one warp per expert e waits for the row cnt[e][0..B), scans it
//            and publishes pre[e][b] (slots of e in CTAs before b) and
//            tot[e] (slots of e).
//   phase 3  every CTA waits for tot[] and its column pre[.][b], scans the
//            totals into expert starts, and each warp places its slots, 32
//            per step: start(e) + pre[e][b] + slots of e in earlier warps of
//            the CTA + earlier steps + lower lanes of the step with the same e
//            (match.any). Every CTA writes its share of the CSR, expert_ids
//            and scale offsets (CTA 0 also the stats); CTA 0 then gathers
//            every CTA's status bits into the status word and advances the
//            call counter.
// Every published value is a 64-bit word tagged with this call's number (see
// tagged_sync.cuh), so a consumer checks the data itself and no fence sits on
// the critical path. Two relaxed counters (CTAs that published their counts,
// rows that published their prefixes) spare the consumers from polling many
// words; each comes in two slots used by alternate calls, and a call zeroes
// the slot of the next one, so nothing is reset from the host. The ids written
// in phase 1 are read back from L2 in phase 3; the [T, K] id matrix is never
// re-read from HBM.
//
// The launch is cooperative, so all CTAs are resident and every wait is met;
// each is bounded all the same (one second). A CTA that gives up records
// MOE_DEVICE_STATUS_SYNC_TIMEOUT and skips the phases that depend on it.
#include "index_device.cuh"
#include "route_device.cuh"
#include "route_staged.cuh"
#include "tagged_sync.cuh"

namespace moe {
namespace {

constexpr int kMaxFusedCtas = 2048;
constexpr int kMinFusedWarps = 8;  // the smallest CTA of the fused kernels
constexpr int kRowPerLane = 8;     // tagged words per lane and pass in phase 2
constexpr size_t kFusedHeaderBytes = 256;

inline size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace: header (status word, call counter) | progress counters (CTAs
// and rows published, two slots each, one 256-byte block per slot) |
// cnt [E][R] | pre [E][R] |
// tot [E] | stat [R], the last four of 64-bit tagged words; R is the CTA
// count rounded up to 4.
struct FusedLayout {
  int64_t row;
  size_t cnt_off, pre_off, tot_off, stat_off, total;
};

FusedLayout fused_layout(int64_t T, int E) {
  FusedLayout L;
  int64_t max_ctas = (T + kMinFusedWarps - 1) / kMinFusedWarps;
  max_ctas = max_ctas < 1 ? 1 : (max_ctas > kMaxFusedCtas ? kMaxFusedCtas : max_ctas);
  L.row = (max_ctas + 3) & ~(int64_t)3;
  const size_t matrix = round256(sizeof(uint64_t) * (size_t)E * (size_t)L.row);
  L.cnt_off = kFusedHeaderBytes + 4 * 256;
  L.pre_off = L.cnt_off + matrix;
  L.tot_off = L.pre_off + matrix;
  L.stat_off = L.tot_off + round256(sizeof(uint64_t) * (size_t)E);
  L.total = L.stat_off + round256(sizeof(uint64_t) * (size_t)L.row);
  return L;
}

struct FusedArgs {
  RouteArgs r;
  IdxArgs x;        // x.ids are r.ids, written in phase 1; x.row = R
  uint64_t* cnt;    // [E][R]
  uint64_t* pre;    // [E][R]
  uint64_t* tot;    // [E]
  uint64_t* stat;   // [R]: each CTA's status bits
  uint32_t* calls;    // header word 1: number of the last call that finished
  uint32_t* counted;  // CTAs whose counts are out: two slots, 256 bytes apart
  uint32_t* scanned;  // rows whose prefixes are out: two slots, 256 bytes apart
};

// Slot of a progress counter used by the call with tag `tag`. Each counter
// word sits in a 256-byte block of its own, so that its pollers and its
// updates load one L2 slice as little as possible.
__device__ __forceinline__ uint32_t* counter(uint32_t* slots, uint32_t tag) {
  return slots + (tag & 1u) * 64u;
}

__device__ __forceinline__ bool wait_slot(uint32_t* slots, uint32_t target, uint32_t tag) {
  return moe::wait_count(counter(slots, tag), target);
}

// Counts one routed slot in the calling warp's row of counts and in the
// CTA's. An id outside [0, E) (possible only for NaN scores) is left out here
// and flagged when the slots are placed.
__device__ __forceinline__ void count_expert(uint32_t* warp_cnt, uint32_t* cta_cnt, int id,
                                             int E) {
  if ((unsigned)id < (unsigned)E) {
    atomicAdd(&warp_cnt[id], 1u);
    atomicAdd(&cta_cnt[id], 1u);
  }
}

// Token ranges: an even split of T over the CTAs, and of a CTA's range over
// its warps.
__device__ __forceinline__ void split(int64_t n0, int64_t n1, int64_t part, int64_t parts,
                                      int64_t& p0, int64_t& p1) {
  p0 = n0 + (n1 - n0) * part / parts;
  p1 = n0 + (n1 - n0) * (part + 1) / parts;
}

// Phase 2: the calling warp waits for the B counts of expert e, scans them and
// publishes the exclusive prefixes and the total. A pass covers 256 CTAs:
// lane l takes the 8 consecutive words l*8 .. l*8+7 of it. Returns false if
// the counts did not all arrive in time.
__device__ bool scan_row(const FusedArgs& f, int e, uint32_t tag) {
  const int B = gridDim.x, R = f.x.row, lane = threadIdx.x & 31;
  const uint64_t* row = f.cnt + (int64_t)e * R;
  uint64_t* out = f.pre + (int64_t)e * R;
  uint32_t carry = 0;
  for (int j0 = 0; j0 < B; j0 += 32 * kRowPerLane) {
    const int jb = j0 + lane * kRowPerLane;
    uint32_t x[kRowPerLane];
    bool ready = false;
    const uint64_t t0 = global_ns();
    for (uint32_t polls = 0;; ++polls) {
      bool mine = true;
#pragma unroll
      for (int u = 0; u < kRowPerLane; ++u) {
        x[u] = 0u;
        if (jb + u < B) {
          const uint64_t w = load_relaxed(row + jb + u);
          mine = mine && has_tag(w, tag);
          x[u] = (uint32_t)w;
        }
      }
      ready = __all_sync(kFullMask, mine);
      if (ready) break;
      const bool expired = polls >= kSyncMaxPolls || global_ns() - t0 > kSyncTimeoutNs;
      if (__shfl_sync(kFullMask, expired, 0)) break;
      __nanosleep(64);
    }
    if (!ready) return false;
    uint32_t sum = 0;
#pragma unroll
    for (int u = 0; u < kRowPerLane; ++u) sum += x[u];
    uint32_t incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(kFullMask, incl, off);
      if (lane >= off) incl += y;
    }
    uint32_t run = carry + incl - sum;
#pragma unroll
    for (int u = 0; u < kRowPerLane; ++u) {
      if (jb + u < B) store_tagged(out + jb + u, tag, run);
      run += x[u];
    }
    carry += __shfl_sync(kFullMask, incl, 31);
  }
  if (lane == 0) store_tagged(f.tot + e, tag, carry);
  __syncwarp();
  if (lane == 0) add_relaxed(counter(f.scanned, tag), 1u);
  return true;
}

// Phase 3 placement of the calling warp's slots [s0, s1), 32 per step: a
// slot of expert e goes to s_base[e] (the CTA's first position for e) +
// warp_off[e] (slots of e before it in this CTA, advanced per step) + the
// lower lanes of its step with the same e.
// Loads the ids of the 32 * kStepsPerWarp slots from c0 on (below s1) that
// the calling warp places in one round: -1 marks a slot past s1 or an id outside [0, E).
__device__ __forceinline__ void load_round(const FusedArgs& f, int64_t c0, int64_t s1,
                                           int (&v)[kStepsPerWarp], bool& bad) {
  const int lane = threadIdx.x & 31, E = f.x.E;
#pragma unroll
  for (int s = 0; s < kStepsPerWarp; ++s) {
    const int64_t i = c0 + s * 32 + lane;
    int id = -1;
    if (i < s1) {
      id = __ldcg(f.x.ids + i);
      if (id < 0 || id >= E) {
        bad = true;
        id = -1;
      }
    }
    v[s] = id;
  }
}

// `v` enters holding the first round's ids (load_round at s0), loaded while
// the CTA waited for the prefixes.
__device__ void place_warp_slots(const FusedArgs& f, int64_t s0, int64_t s1,
                                 const uint32_t* s_base, uint32_t* warp_off,
                                 int (&v)[kStepsPerWarp], bool& bad, bool& overflow) {
  const IdxArgs& a = f.x;
  const int lane = threadIdx.x & 31;
  const unsigned lower = lanemask_lt();
  for (int64_t c0 = s0; c0 < s1; c0 += 32 * kStepsPerWarp) {
    if (c0 != s0) load_round(f, c0, s1, v, bad);
#pragma unroll
    for (int s = 0; s < kStepsPerWarp; ++s) {
      if (c0 + s * 32 >= s1) break;  // warp-uniform
      const int64_t i = c0 + s * 32 + lane;
      const unsigned peers = __match_any_sync(kFullMask, v[s]);
      uint32_t pos = 0xFFFFFFFFu;
      if (v[s] >= 0) pos = s_base[v[s]] + warp_off[v[s]] + (uint32_t)__popc(peers & lower);
      __syncwarp();
      if (v[s] >= 0 && lane == __ffs(peers) - 1) warp_off[v[s]] += (uint32_t)__popc(peers);
      __syncwarp();
      if (i < s1) {
        a.restore_token_order[i] = pos;
        if (v[s] >= 0) {
          if (pos < a.N)
            a.token_expert_order[pos] = (uint32_t)i;
          else
            overflow = true;  // impossible with consistent counts; reported, never written
        }
      }
    }
  }
}

// Everything after routing. s_warp [warps][E] holds each warp's expert counts
// for its tokens [tw0, tw1) and s_cnt [E] the CTA's; `work` is at least 5E
// words of shared scratch. `tag` is this call's number.
__device__ void build_index(const FusedArgs& f, uint32_t* s_warp, const uint32_t* s_cnt,
                            uint32_t* work, int64_t tw0, int64_t tw1, uint32_t tag) {
  __shared__ uint32_t s_bits;
  __shared__ int s_flag;
  const IdxArgs& a = f.x;
  const int E = a.E, B = gridDim.x, b = blockIdx.x, R = a.row;
  const int nwarps = blockDim.x >> 5, warp = threadIdx.x >> 5;
  uint32_t* s_tot = work;          // slots of each expert
  uint32_t* s_pre = work + E;      // slots of each expert in CTAs before this one
  uint32_t* s_start = work + 2 * E;
  uint32_t* s_act = work + 3 * E;
  uint32_t* s_pad = work + 4 * E;
  if (threadIdx.x == 0) s_bits = 0;
  // phase 1 result: this CTA's count of each expert (the caller synchronised)
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    store_tagged(f.cnt + (int64_t)e * R + b, tag, s_cnt[e]);
  __syncthreads();
  if (threadIdx.x == 0) add_relaxed(counter(f.counted, tag), 1u);
  // per-warp offsets within the CTA (needed in phase 3)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    uint32_t run = 0;
    for (int w = 0; w < nwarps; ++w) {
      const uint32_t c = s_warp[w * E + e];
      s_warp[w * E + e] = run;
      run += c;
    }
  }
  // phase 2, in the CTAs that own rows: one thread waits until every CTA has
  // published its counts (few pollers keep the counter's L2 slice free for
  // the routing traffic of the CTAs still at work)
  bool ok = true;
  if (b * nwarps < E) {
    if (threadIdx.x == 0) s_flag = wait_slot(f.counted, (uint32_t)B, tag);
    __syncthreads();
    ok = s_flag != 0;
    for (int e = b * nwarps + warp; e < E; e += B * nwarps) ok = ok && scan_row(f, e, tag);
    __syncthreads();
  }
  // this warp's first round of ids, loaded while the other CTAs finish
  const int64_t K = f.r.K;
  bool bad = false, overflow = false;
  int v[kStepsPerWarp];
  load_round(f, tw0 * K, tw1 * K, v, bad);
  // phase 3: wait for every row, then read the totals and this CTA's prefixes
  if (threadIdx.x == 0) s_flag = wait_slot(f.scanned, (uint32_t)E, tag);
  __syncthreads();
  ok = ok && s_flag != 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    uint32_t t = 0, pr = 0;
    ok = ok && wait_tagged(f.tot + e, tag, t) && wait_tagged(f.pre + (int64_t)e * R + b, tag, pr);
    s_tot[e] = t;
    s_pre[e] = pr;
  }
  ok = __syncthreads_and(ok);
  if (ok) {
    const TableSums sums = scan_expert_table(s_tot, s_start, s_act, s_pad, E);
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_pre[e] += s_start[e];
    __syncthreads();
    place_warp_slots(f, tw0 * K, tw1 * K, s_pre, s_warp + warp * E, v, bad, overflow);
    write_table_share(a, s_tot, s_start, s_act, s_pad, sums);
  }
  // this CTA's status bits
  const int any_bad = __syncthreads_or(bad);
  const int any_overflow = __syncthreads_or(overflow);
  if (threadIdx.x == 0) {
    uint32_t bits = ok ? 0u : MOE_DEVICE_STATUS_SYNC_TIMEOUT;
    if (any_bad) bits |= MOE_DEVICE_STATUS_BAD_EXPERT_ID;
    if (any_overflow) bits |= MOE_DEVICE_STATUS_SYNC_STATE;
    store_tagged(f.stat + b, tag, bits);
  }
  if (b != 0) return;
  // CTA 0: gather every CTA's bits into the status word, then count the call
  for (int j = threadIdx.x; j < B; j += blockDim.x) {
    uint32_t bits = 0;
    if (!wait_tagged(f.stat + j, tag, bits)) bits = MOE_DEVICE_STATUS_SYNC_TIMEOUT;
    if (bits) atomicOr(&s_bits, bits);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    *a.status = s_bits;
    *f.calls = tag;
  }
}

// This call's tag: one more than the last finished call's. 0 is never a tag,
// so a zero-filled workspace never looks ready; after 0xFFFFFFFF comes 2, not
// 1, so consecutive tags keep alternating in parity, which picks their
// counter slot. CTA 0 also zeroes the counter slot of the next call; the
// previous user of that slot, the call before this one, has finished.
__device__ __forceinline__ uint32_t call_tag(const FusedArgs& f) {
  __shared__ uint32_t s_tag;
  if (threadIdx.x == 0) {
    uint32_t t = load_relaxed(f.calls) + 1u;
    t = t == 0u ? 2u : t;
    s_tag = t;
    if (blockIdx.x == 0) {
      *counter(f.counted, t + 1u) = 0u;
      *counter(f.scanned, t + 1u) = 0u;
    }
  }
  __syncthreads();
  return s_tag;
}

// Shared memory of both kernels: s_warp [warps][E] | s_cnt [E] | work.
struct FusedSmem {
  uint32_t* s_warp;
  uint32_t* s_cnt;
  uint32_t* work;
};

__device__ __forceinline__ FusedSmem fused_smem_layout(uint32_t* dyn, int warps, int E) {
  FusedSmem m;
  m.s_warp = dyn;
  m.s_cnt = dyn + warps * E;
  m.work = m.s_cnt + E;
  return m;
}

// CTA size of the fused kernels: as many warps as the registers of one SM
// allow at the kernel's register count (64, 128 or 255 per thread), so that
// one CTA per SM carries the router's full warp count and the count matrix
// has as few CTA columns as possible.
template <int C>
__host__ __device__ constexpr int warp_kernel_warps() {
  return C <= 8 ? 32 : (C <= 16 ? 16 : 8);
}
template <int EP>
__host__ __device__ constexpr int thread_kernel_warps() {
  return EP <= 8 ? 32 : (EP <= 16 ? 16 : 8);
}

template <int C, bool kVec, bool kSoftmax>
__global__ void __launch_bounds__(warp_kernel_warps<C>() * 32, 1)
    route_index_warp_kernel(const FusedArgs f) {
  extern __shared__ __align__(16) uint32_t dyn[];
  constexpr int kWarps = warp_kernel_warps<C>();
  const int E = f.x.E, warp = threadIdx.x >> 5;
  const FusedSmem m = fused_smem_layout(dyn, kWarps, E);
  wait_for_prior_grid();
  for (int i = threadIdx.x; i < (kWarps + 1) * E; i += blockDim.x) m.s_warp[i] = 0;
  const uint32_t tag = call_tag(f);  // includes a block barrier
  int64_t t0, t1, tw0, tw1;
  split(0, f.r.T, blockIdx.x, gridDim.x, t0, t1);
  split(t0, t1, warp, kWarps, tw0, tw1);
  uint32_t* warp_cnt = m.s_warp + warp * E;
  uint32_t* cta_cnt = m.s_cnt;
  if (tw0 < tw1) {
    // the work area holds the generic group layout's scores during routing
    route_tokens_warp<C, kVec, kSoftmax>(f.r, tw0, tw1, 1,
                               reinterpret_cast<float*>(m.work) + warp * f.r.warp_smem_words,
                               [&](int64_t, int, int id) { count_expert(warp_cnt, cta_cnt, id, E); });
  }
  __syncthreads();
  build_index(f, m.s_warp, m.s_cnt, m.work, tw0, tw1, tag);
}

template <int EP, bool kVec>
__global__ void __launch_bounds__(thread_kernel_warps<EP>() * 32, 1)
    route_index_thread_kernel(const FusedArgs f) {
  extern __shared__ __align__(16) uint32_t dyn[];
  constexpr int kWarps = thread_kernel_warps<EP>();
  const int E = f.x.E, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const FusedSmem m = fused_smem_layout(dyn, kWarps, E);
  wait_for_prior_grid();
  for (int i = threadIdx.x; i < (kWarps + 1) * E; i += blockDim.x) m.s_warp[i] = 0;
  const uint32_t tag = call_tag(f);
  int64_t t0, t1, tw0, tw1;
  split(0, f.r.T, blockIdx.x, gridDim.x, t0, t1);
  split(t0, t1, warp, kWarps, tw0, tw1);
  uint32_t* warp_cnt = m.s_warp + warp * E;
  uint32_t* cta_cnt = m.s_cnt;
  if (tw0 + lane < tw1) {
    route_tokens_thread<EP, kVec>(f.r, tw0 + lane, tw1, 32,
                                  [&](int64_t, int, int id) { count_expert(warp_cnt, cta_cnt, id, E); });
  }
  __syncthreads();
  build_index(f, m.s_warp, m.s_cnt, m.work, tw0, tw1, tag);
}

// Launches `k` cooperatively with `warps` warps per CTA on min(T /
// tokens_per_cta, resident CTAs) CTAs, with programmatic stream
// serialisation when the CUDA driver accepts both.
template <typename Kernel>
moe_status_t launch_fused(Kernel k, FusedArgs f, int warps, int64_t tokens_per_cta, size_t smem,
                          cudaStream_t stream) {
  // above 40 KB of dynamic shared memory, opt in past the default 48 KB limit
  // (the kernels also hold a few hundred bytes of static shared memory)
  if (smem > 40 * 1024 && set_dynamic_smem((const void*)k, smem) != MOE_OK) return MOE_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, warps * 32, smem) !=
          cudaSuccess ||
      per_sm < 1)
    return MOE_ERR_UNSUPPORTED;
  int64_t cap = (int64_t)device_info().sm_count * per_sm;
  if (cap > kMaxFusedCtas) cap = kMaxFusedCtas;
  int64_t want = (f.r.T + tokens_per_cta - 1) / tokens_per_cta;
  if (want < 1) want = 1;
  const int grid = (int)(want < cap ? want : cap);
  if ((grid + 3) / 4 * 4 > f.x.row) return MOE_ERR_WORKSPACE;  // never: the layout bounds it
  f.x.num_blocks = grid;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(warps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, k, f) != cudaSuccess) {
    cudaGetLastError();
    cfg.numAttrs = 1;  // cooperative alone
    if (cudaLaunchKernelEx(&cfg, k, f) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  }
  return launch_status();
}

// Dynamic shared memory of a fused CTA with `warps` warps.
size_t fused_smem(const RoutePlan& p, int warps) {
  const size_t E = (size_t)p.a.E;
  size_t work = 5 * E;  // totals, prefixes, starts, active and padded offsets
  const size_t routing = route_warp_smem(p, warps) / sizeof(uint32_t);
  if (work < routing) work = routing;  // the routing warps' shared memory
  return sizeof(uint32_t) * ((size_t)(warps + 1) * E + work);
}

template <int C, bool kSoftmax>
moe_status_t launch_fused_warp_fn(const RoutePlan& p, const FusedArgs& f, cudaStream_t stream) {
  constexpr int W = warp_kernel_warps<C>();
  const size_t smem = fused_smem(p, W);
  if constexpr (C % 4 == 0) {
    if (p.vec)
      return launch_fused(route_index_warp_kernel<C, true, kSoftmax>, f, W, W, smem, stream);
  }
  return launch_fused(route_index_warp_kernel<C, false, kSoftmax>, f, W, W, smem, stream);
}

template <int C>
moe_status_t launch_fused_warp(const RoutePlan& p, const FusedArgs& f, cudaStream_t stream) {
  if (p.a.score_fn == MOE_SCORES_SOFTMAX) return launch_fused_warp_fn<C, true>(p, f, stream);
  return launch_fused_warp_fn<C, false>(p, f, stream);
}

template <int EP>
moe_status_t launch_fused_thread(const RoutePlan& p, const FusedArgs& f, cudaStream_t stream) {
  constexpr int W = thread_kernel_warps<EP>();
  const size_t smem = fused_smem(p, W);
  if (p.vec)
    return launch_fused(route_index_thread_kernel<EP, true>, f, W, 32 * W, smem, stream);
  return launch_fused(route_index_thread_kernel<EP, false>, f, W, 32 * W, smem, stream);
}

// ---------------------------------------------------------------- three-kernel path
// moe_route_index: the router counts its own output, so the index build starts
// at the row prefixes. Slot i = t*K+k of expert e adds one to counts[e][i /
// 1024] (a relaxed atomic: integer sums do not depend on the order); the
// rows kernel turns each expert's row into prefixes and totals; the scatter
// CTA of chunk b places its 1024 slots and leaves column b zero again for the
// next call. No CTA waits on another: the kernel boundaries order the phases.

struct CountRouteArgs {
  RouteArgs r;
  uint32_t* counts;  // [E][row], zero on entry; nullptr: route without counting
  int row;
};

// Adds one to the count word of (id, slot's chunk). The lanes of the warp
// that are here together and add to the same word combine first (one atomic
// of their number): with few or skewed experts, hundreds of slots of a chunk
// land on the same word, and serialised atomics on it cost more than the
// routing. Which lanes combine does not change the sum.
__device__ __forceinline__ void count_slot(uint32_t* counts, int row, int E, int64_t slot,
                                           int id) {
  if (counts == nullptr || (unsigned)id >= (unsigned)E) return;
  uint32_t* word = counts + (int64_t)id * row + slot / kSlotsPerCta;
  const unsigned here = __activemask();
  const unsigned same = __match_any_sync(here, reinterpret_cast<unsigned long long>(word));
  if ((int)(threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(word, (uint32_t)__popc(same));
}

__device__ __forceinline__ void count_slot(const CountRouteArgs& c, int64_t slot, int id) {
  count_slot(c.counts, c.row, c.r.E, slot, id);
}

template <int C, bool kVec, bool kSoftmax>
__global__ void __launch_bounds__(kRouteThreads, C <= 8 ? 4 : 2)
    route_count_warp_kernel(const CountRouteArgs c) {
  extern __shared__ float dyn_smem[];  // kRouteWarps * c.r.warp_smem_words
  wait_for_prior_grid();
  const int warp = threadIdx.x >> 5;
  const int64_t K = c.r.K;
  route_tokens_warp<C, kVec, kSoftmax>(
      c.r, (int64_t)blockIdx.x * kRouteWarps + warp, c.r.T, (int64_t)gridDim.x * kRouteWarps,
      dyn_smem + warp * c.r.warp_smem_words,
      [&](int64_t t, int k, int id) { count_slot(c, t * K + k, id); });
}

template <int L, bool kGroups, bool kSoftmax>
__global__ void __launch_bounds__(kRouteThreads, 3) route_count_seg_kernel(const CountRouteArgs c) {
  extern __shared__ float dyn_smem[];  // softmax loader: c.r.warp_smem_words per warp
  __shared__ __align__(16) float s_bias[kSegBiasStride * (MOE_MAX_EXPERTS / kSegKeys)];
  __shared__ uint64_t s_cand[kRouteWarps * (32 / L) * kSegCand];
  __shared__ int s_slot[kRouteWarps * (32 / L) * kSegTop];
  wait_for_prior_grid();
  if (threadIdx.x < 32) stage_seg_bias(c.r, s_bias);
  __syncthreads();
  const int warps = blockDim.x >> 5;
  const int64_t K = c.r.K;
  const int warp = threadIdx.x >> 5;
  route_tokens_seg<L, kGroups, kSoftmax>(c.r, s_bias, s_cand + warp * (32 / L) * kSegCand,
                               s_slot + warp * (32 / L) * kSegTop,
                               kSoftmax ? dyn_smem + warp * c.r.warp_smem_words : nullptr,
                               (int64_t)blockIdx.x * warps + warp,
                               (int64_t)gridDim.x * warps,
                               [&](int64_t t, int k, int id) { count_slot(c, t * K + k, id); });
}

// kKc: K fixed at compile time (8, the common case), or 0 for any K <= 8.
// kSigmoid / kSoftmax: the score loader (the softmax loader with K = 8 only).
template <int G, bool kSigmoid, int kKc, bool kSoftmax = false>
__global__ void __launch_bounds__(kStagedThreadsMax, 1)
    route_count_staged_kernel(const CountRouteArgs c, const StagedSplit sp) {
  extern __shared__ __align__(128) char staged_smem_buf[];
  wait_for_prior_grid();
  uint32_t* const counts = c.counts;
  const int row = c.row, E = c.r.E;
  const int64_t K = c.r.K;
  route_tokens_staged<kStagedR, G / kStagedR, kSigmoid, kKc, kSoftmax>(
      c.r, staged_smem_buf, sp,
      [=](int64_t t, int k, int id) { count_slot(counts, row, E, t * K + k, id); });
}

template <int EP, bool kVec>
__global__ void __launch_bounds__(kRouteThreads) route_count_thread_kernel(const CountRouteArgs c) {
  wait_for_prior_grid();
  const int64_t K = c.r.K;
  route_tokens_thread<EP, kVec>(c.r, (int64_t)blockIdx.x * blockDim.x + threadIdx.x, c.r.T,
                                (int64_t)gridDim.x * blockDim.x,
                                [&](int64_t t, int k, int id) { count_slot(c, t * K + k, id); });
}

// Workspace of the three-kernel path: header (word 0: status) | totals
// [MOE_MAX_EXPERTS] | counts [E][row] ... prefixes [E][row] at the END of the
// caller's workspace. Every call leaves its counts zero, the counts start at a
// fixed place and the prefixes end at the workspace's end; since each call's
// counts and prefixes both fit, no call's counts reach words that another
// call's prefixes left nonzero, whatever the shapes and their order.
struct SplitLayout {
  int64_t num_blocks, row;
  size_t totals_off, counts_off, matrix_bytes, total;
};

SplitLayout split_layout(int64_t N, int E) {
  SplitLayout L;
  L.num_blocks = (N + kSlotsPerCta - 1) / kSlotsPerCta;
  if (L.num_blocks < 1) L.num_blocks = 1;
  L.row = (L.num_blocks + 3) & ~(int64_t)3;
  L.totals_off = kFusedHeaderBytes;
  L.counts_off = L.totals_off + sizeof(uint32_t) * MOE_MAX_EXPERTS;
  L.matrix_bytes = round256(sizeof(uint32_t) * (size_t)E * (size_t)L.row);
  L.total = L.counts_off + 2 * L.matrix_bytes;
  return L;
}

template <typename Kernel, typename Args>
moe_status_t launch_counting_router(Kernel k, const Args& args, int64_t T, int64_t tokens_per_cta,
                                    size_t smem, cudaStream_t stream,
                                    int threads = kRouteThreads) {
  if (smem > 40 * 1024 && set_dynamic_smem((const void*)k, smem) != MOE_OK) return MOE_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (T + tokens_per_cta - 1) / tokens_per_cta;
  const int64_t cap = (int64_t)device_info().sm_count * per_sm;
  const int grid = (int)(want < cap ? want : cap);
  return launch(k, grid, threads, smem, stream, args);
}

template <int C, bool kSoftmax>
moe_status_t launch_count_warp_fn(const RoutePlan& p, const CountRouteArgs& c,
                                  cudaStream_t stream) {
  const size_t smem = route_warp_smem(p, kRouteWarps);
  if constexpr (C % 4 == 0) {
    if (p.vec)
      return launch_counting_router(route_count_warp_kernel<C, true, kSoftmax>, c, c.r.T,
                                    kRouteWarps, smem, stream);
  }
  return launch_counting_router(route_count_warp_kernel<C, false, kSoftmax>, c, c.r.T,
                                kRouteWarps, smem, stream);
}

template <int C>
moe_status_t launch_count_warp(const RoutePlan& p, const CountRouteArgs& c, cudaStream_t stream) {
  if (p.a.score_fn == MOE_SCORES_SOFTMAX) return launch_count_warp_fn<C, true>(p, c, stream);
  return launch_count_warp_fn<C, false>(p, c, stream);
}

template <int EP>
moe_status_t launch_count_thread(const RoutePlan& p, const CountRouteArgs& c,
                                 cudaStream_t stream) {
  if (p.vec)
    return launch_counting_router(route_count_thread_kernel<EP, true>, c, c.r.T, kRouteThreads,
                                  0, stream);
  return launch_counting_router(route_count_thread_kernel<EP, false>, c, c.r.T, kRouteThreads, 0,
                                stream);
}

template <int L, bool kSoftmax>
moe_status_t launch_count_seg_fn(const RoutePlan& p, const CountRouteArgs& c,
                                 cudaStream_t stream) {
  const int warps = seg_warps_per_cta(c.r.T, L, device_info().sm_count);
  const int64_t tokens_per_cta = (int64_t)warps * (32 / L);
  const size_t smem = kSoftmax ? route_warp_smem(p, warps) : 0;
  if (p.a.group_mode == kGroupsAllKept)
    return launch_counting_router(route_count_seg_kernel<L, false, kSoftmax>, c, c.r.T,
                                  tokens_per_cta, smem, stream, 32 * warps);
  return launch_counting_router(route_count_seg_kernel<L, true, kSoftmax>, c, c.r.T,
                                tokens_per_cta, smem, stream, 32 * warps);
}

template <int L>
moe_status_t launch_count_seg(const RoutePlan& p, const CountRouteArgs& c, cudaStream_t stream) {
  if (p.a.score_fn == MOE_SCORES_SOFTMAX) return launch_count_seg_fn<L, true>(p, c, stream);
  return launch_count_seg_fn<L, false>(p, c, stream);
}

template <int G, bool kSigmoid>
moe_status_t launch_count_staged_fn(const CountRouteArgs& c, cudaStream_t stream) {
  constexpr int kTok = 32 / kStagedR;
  if (c.r.K == kSegTop)
    return launch_staged(route_count_staged_kernel<G, kSigmoid, kSegTop>, c, c.r.T, c.r.E, kTok,
                         stream);
  return launch_staged(route_count_staged_kernel<G, kSigmoid, 0>, c, c.r.T, c.r.E, kTok, stream);
}

template <int G>
moe_status_t launch_count_staged(const RoutePlan& p, const CountRouteArgs& c,
                                 cudaStream_t stream) {
  constexpr int kTok = 32 / kStagedR;
  if (p.a.score_fn == MOE_SCORES_SOFTMAX)  // K = 8 (plan_route)
    return launch_staged(route_count_staged_kernel<G, false, kSegTop, true>, c, c.r.T, c.r.E,
                         kTok, stream);
  if (p.a.score_fn == MOE_SCORES_SIGMOID) return launch_count_staged_fn<G, true>(c, stream);
  return launch_count_staged_fn<G, false>(c, stream);
}

moe_status_t launch_counting_route(const RoutePlan& p, const CountRouteArgs& c,
                                   cudaStream_t stream) {
  switch (p.staged) {
    case 4: return launch_count_staged<4>(p, c, stream);
    case 8: return launch_count_staged<8>(p, c, stream);
    case 16: return launch_count_staged<16>(p, c, stream);
    default: break;
  }
  switch (p.seg) {
    case 2: return launch_count_seg<2>(p, c, stream);
    case 4: return launch_count_seg<4>(p, c, stream);
    case 8: return launch_count_seg<8>(p, c, stream);
    case 16: return launch_count_seg<16>(p, c, stream);
    case 32: return launch_count_seg<32>(p, c, stream);
    default: break;
  }
  switch (p.C) {
    case 0:
      if (p.EP == 8) return launch_count_thread<8>(p, c, stream);
      if (p.EP == 16) return launch_count_thread<16>(p, c, stream);
      return launch_count_thread<32>(p, c, stream);
    case 2: return launch_count_warp<2>(p, c, stream);
    case 4: return launch_count_warp<4>(p, c, stream);
    case 8: return launch_count_warp<8>(p, c, stream);
    case 16: return launch_count_warp<16>(p, c, stream);
    default: return launch_count_warp<32>(p, c, stream);
  }
}

// The rows and scatter kernels (index_device.cuh) after the counting router.
moe_status_t launch_rows_scatter(const IdxArgs& a, cudaStream_t stream) {
  const size_t scatter_smem = sizeof(uint32_t) * (size_t)(kIdxWarps + 5) * a.E;
  if (scatter_smem > 40 * 1024 &&
      set_dynamic_smem((const void*)idx_scatter_kernel<kBasesFromCounts>, scatter_smem) != MOE_OK)
    return MOE_ERR_CUDA;
  const moe_status_t st = launch(idx_rows_kernel, (a.E + kRowsWarps - 1) / kRowsWarps,
                                 kRowsWarps * 32, 0, stream, a);
  if (st != MOE_OK) return st;
  return launch(idx_scatter_kernel<kBasesFromCounts>, a.num_blocks, kIdxThreads, scatter_smem,
                stream, a);
}

// Checks shared by both entry points; fills the router plan.
moe_status_t check_route_index(int32_t* expert_indices, float* expert_weights,
                               uint32_t* token_expert_order, uint32_t* expert_start_indices,
                               uint32_t* restore_token_order, int32_t* expert_ids,
                               uint32_t* expert_usage_stats, const float* expert_scores,
                               const float* expert_bias, int64_t num_tokens,
                               int32_t n_routed_experts, int32_t n_experts_per_tok,
                               int32_t n_groups, int32_t topk_group, int32_t norm_weights,
                               float routed_scaling_factor, int32_t score_fn,
                               uint32_t* scales_offset_p, RoutePlan* p) {
  moe_status_t st = plan_route(expert_indices, expert_weights, expert_scores, expert_bias,
                               num_tokens, n_routed_experts, n_experts_per_tok, n_groups,
                               topk_group, norm_weights, routed_scaling_factor, score_fn, p);
  if (st != MOE_OK) return st;
  const int64_t T = num_tokens, E = n_routed_experts;
  const int64_t N = T * n_experts_per_tok;
  if (N > (int64_t)0xFFFFFFFEu) return MOE_ERR_UNSUPPORTED;
  if (scales_offset_p != nullptr && N + (int64_t)(kScaleRowAlign - 1) * E > (int64_t)0xFFFFFFFFu)
    return MOE_ERR_UNSUPPORTED;
  if (!expert_start_indices || !expert_ids || !expert_usage_stats) return MOE_ERR_NULL_PTR;
  if (T > 0) {
    st = check_route_pointers(p->a);
    if (st != MOE_OK) return st;
    if (!token_expert_order || !restore_token_order) return MOE_ERR_NULL_PTR;
  }
  if (!aligned(token_expert_order, 4) || !aligned(expert_start_indices, 4) ||
      !aligned(restore_token_order, 4) || !aligned(expert_ids, 4) ||
      !aligned(expert_usage_stats, 4) || !aligned(scales_offset_p, 4))
    return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_route_index_single_launch_workspace_size(int64_t num_tokens,
                                                                int32_t n_routed_experts) {
  if (num_tokens < 0 || n_routed_experts < 1 || n_routed_experts > MOE_MAX_EXPERTS) return 0;
  return moe::fused_layout(num_tokens, n_routed_experts).total;
}

extern "C" moe_status_t moe_route_index_single_launch(
    int32_t* expert_indices, float* expert_weights, uint32_t* token_expert_order,
    uint32_t* expert_start_indices, uint32_t* restore_token_order, int32_t* expert_ids,
    uint32_t* expert_usage_stats, const float* expert_scores, const float* expert_bias,
    int64_t num_tokens, int32_t n_routed_experts, int32_t n_experts_per_tok, int32_t n_groups,
    int32_t topk_group, int32_t norm_weights, float routed_scaling_factor,
    moe_score_fn_t score_fn, void* workspace, size_t workspace_bytes, uint32_t* scales_offset_p,
    cudaStream_t stream) {
  using namespace moe;
  RoutePlan p;
  moe_status_t st = check_route_index(
      expert_indices, expert_weights, token_expert_order, expert_start_indices,
      restore_token_order, expert_ids, expert_usage_stats, expert_scores, expert_bias, num_tokens,
      n_routed_experts, n_experts_per_tok, n_groups, topk_group, norm_weights,
      routed_scaling_factor, score_fn, scales_offset_p, &p);
  if (st != MOE_OK) return st;
  const int64_t T = num_tokens, E = n_routed_experts;
  const int64_t N = T * n_experts_per_tok;
  const FusedLayout L = fused_layout(T, (int)E);
  if (!workspace || workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MOE_ERR_MISALIGNED;

  char* ws = static_cast<char*>(workspace);
  uint32_t* header = reinterpret_cast<uint32_t*>(ws);
  FusedArgs f{};
  f.r = p.a;
  f.x.ids = expert_indices;
  f.x.token_expert_order = token_expert_order;
  f.x.expert_start_indices = expert_start_indices;
  f.x.restore_token_order = restore_token_order;
  f.x.expert_ids = expert_ids;
  f.x.stats = expert_usage_stats;
  f.x.status = header;
  f.x.flags = nullptr;
  f.x.counts = nullptr;
  f.x.totals = nullptr;
  f.x.prefix = nullptr;
  f.x.counts_from_router = 0;
  f.x.scales_offset = scales_offset_p;
  f.x.N = (uint32_t)N;
  f.x.E = (int)E;
  f.x.num_blocks = 0;  // set at launch
  f.x.row = (int)L.row;
  f.cnt = reinterpret_cast<uint64_t*>(ws + L.cnt_off);
  f.pre = reinterpret_cast<uint64_t*>(ws + L.pre_off);
  f.tot = reinterpret_cast<uint64_t*>(ws + L.tot_off);
  f.stat = reinterpret_cast<uint64_t*>(ws + L.stat_off);
  f.calls = header + 1;
  f.counted = reinterpret_cast<uint32_t*>(ws + kFusedHeaderBytes);
  f.scanned = reinterpret_cast<uint32_t*>(ws + kFusedHeaderBytes + 2 * 256);

  switch (p.C) {
    case 0:
      if (p.EP == 8) return launch_fused_thread<8>(p, f, stream);
      if (p.EP == 16) return launch_fused_thread<16>(p, f, stream);
      return launch_fused_thread<32>(p, f, stream);
    case 2: return launch_fused_warp<2>(p, f, stream);
    case 4: return launch_fused_warp<4>(p, f, stream);
    case 8: return launch_fused_warp<8>(p, f, stream);
    case 16: return launch_fused_warp<16>(p, f, stream);
    default: return launch_fused_warp<32>(p, f, stream);
  }
}

extern "C" size_t moe_route_index_workspace_size(int64_t num_tokens, int32_t n_routed_experts,
                                                 int32_t n_experts_per_tok) {
  if (num_tokens < 0 || n_routed_experts < 1 || n_routed_experts > MOE_MAX_EXPERTS ||
      n_experts_per_tok < 1 || n_experts_per_tok > MOE_MAX_EXPERTS_PER_TOK)
    return 0;
  return moe::split_layout(num_tokens * n_experts_per_tok, n_routed_experts).total;
}

extern "C" moe_status_t moe_route_index(
    int32_t* expert_indices, float* expert_weights, uint32_t* token_expert_order,
    uint32_t* expert_start_indices, uint32_t* restore_token_order, int32_t* expert_ids,
    uint32_t* expert_usage_stats, const float* expert_scores, const float* expert_bias,
    int64_t num_tokens, int32_t n_routed_experts, int32_t n_experts_per_tok, int32_t n_groups,
    int32_t topk_group, int32_t norm_weights, float routed_scaling_factor,
    moe_score_fn_t score_fn, void* workspace, size_t workspace_bytes, uint32_t* scales_offset_p,
    cudaStream_t stream) {
  using namespace moe;
  RoutePlan p;
  moe_status_t st = check_route_index(
      expert_indices, expert_weights, token_expert_order, expert_start_indices,
      restore_token_order, expert_ids, expert_usage_stats, expert_scores, expert_bias, num_tokens,
      n_routed_experts, n_experts_per_tok, n_groups, topk_group, norm_weights,
      routed_scaling_factor, score_fn, scales_offset_p, &p);
  if (st != MOE_OK) return st;
  const int64_t T = num_tokens, N = T * n_experts_per_tok;
  const SplitLayout L = split_layout(N, n_routed_experts);
  if (!workspace || workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MOE_ERR_MISALIGNED;

  char* ws = static_cast<char*>(workspace);
  IdxArgs x{};
  x.ids = expert_indices;
  x.token_expert_order = token_expert_order;
  x.expert_start_indices = expert_start_indices;
  x.restore_token_order = restore_token_order;
  x.expert_ids = expert_ids;
  x.stats = expert_usage_stats;
  x.status = reinterpret_cast<uint32_t*>(ws);
  x.flags = nullptr;
  x.counts = reinterpret_cast<uint32_t*>(ws + L.counts_off);
  x.totals = reinterpret_cast<uint32_t*>(ws + L.totals_off);
  // prefixes at the end of the caller's workspace, 256-byte aligned
  x.prefix = reinterpret_cast<uint32_t*>(ws + (workspace_bytes - L.matrix_bytes) / 256 * 256);
  x.scales_offset = scales_offset_p;
  x.counts_from_router = 1;
  x.N = (uint32_t)N;
  x.E = n_routed_experts;
  x.num_blocks = (int)L.num_blocks;
  x.row = (int)L.row;

  CountRouteArgs c{};
  c.r = p.a;
  c.counts = L.num_blocks > 1 ? x.counts : nullptr;
  c.row = (int)L.row;
  if (T > 0) {
    st = launch_counting_route(p, c, stream);
    if (st != MOE_OK) return st;
  }
  if (L.num_blocks > 1) return launch_rows_scatter(x, stream);
  // one CTA places every slot (and writes the status word) without counts
  const size_t smem = sizeof(uint32_t) * (size_t)(kIdxWarps + 5) * x.E;
  if (smem > 40 * 1024 &&
      set_dynamic_smem((const void*)idx_scatter_kernel<kBasesSingleCta>, smem) != MOE_OK)
    return MOE_ERR_CUDA;
  return launch(idx_scatter_kernel<kBasesSingleCta>, 1, kIdxThreads, smem, stream, x);
}
