// Device code of the expert index builder (page "moe_create_indices"),
// shared by the index kernels and the fused router + index kernel: the
// argument block, the blocked scan of the expert totals and the expert table
// (compact CSR, expert_ids, usage stats, aligned scale offsets).
#pragma once

#include "common.cuh"

namespace moe {
namespace {

constexpr int kIdxThreads = 256;
constexpr int kIdxWarps = kIdxThreads / 32;
constexpr int kStepsPerWarp = 4;
constexpr int kSlotsPerWarp = 32 * kStepsPerWarp;
constexpr int kSlotsPerCta = kIdxWarps * kSlotsPerWarp;  // 1024
constexpr uint32_t kScaleRowAlign = MOE_SCALES_ROW_ALIGNMENT;
constexpr int kRowsWarps = 8;  // rows kernel: warps per CTA, one expert each

struct IdxArgs {
  const int32_t* ids;
  uint32_t* token_expert_order;
  uint32_t* expert_start_indices;
  uint32_t* restore_token_order;
  int32_t* expert_ids;
  uint32_t* stats;
  uint32_t* status;  // workspace word 0
  uint32_t* flags;   // [num_blocks]
  uint32_t* counts;  // [E][row] counts of each expert in each CTA chunk
  uint32_t* prefix;  // [E][row]: the rows kernel's prefixes (may be `counts` itself)
  uint32_t* totals;  // [E]: slots of each expert
  uint32_t* scales_offset;  // optional [E+1]: 128-row aligned per-expert offsets
  int counts_from_router;   // counts accumulated by the router (see idx_rows_kernel)
  uint32_t N;
  int E;
  int num_blocks;
  int row;
};

// Sums that the expert table needs besides the per-expert arrays.
struct TableSums {
  uint32_t slots, active, padded_total, max_count;
};

// From tot[0..E) (shared memory), every thread of the block computes, in one
// pass of a blocked scan: start[e] (slots before expert e), act[e] (active
// experts before e), pad[e] (128-row padded slots before e), and the sums.
__device__ TableSums scan_expert_table(const uint32_t* tot, uint32_t* start, uint32_t* act,
                                       uint32_t* pad, int E) {
  __shared__ uint4 w_sum[32];
  __shared__ uint4 s_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  const int per = (E + (int)blockDim.x - 1) / (int)blockDim.x;
  const int beg = min((int)threadIdx.x * per, E), end = min(beg + per, E);
  uint32_t st = 0, ac = 0, pd = 0, mx = 0;
  for (int e = beg; e < end; ++e) {
    const uint32_t c = tot[e];
    st += c;
    ac += c > 0u;
    pd += (c + (kScaleRowAlign - 1)) / kScaleRowAlign * kScaleRowAlign;
    mx = max(mx, c);
  }
  uint32_t ist = st, iac = ac, ipd = pd;  // inclusive warp scans
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t a0 = __shfl_up_sync(kFullMask, ist, off);
    const uint32_t a1 = __shfl_up_sync(kFullMask, iac, off);
    const uint32_t a2 = __shfl_up_sync(kFullMask, ipd, off);
    if (lane >= off) {
      ist += a0;
      iac += a1;
      ipd += a2;
    }
  }
  const uint32_t wmax = __reduce_max_sync(kFullMask, mx);
  if (lane == 31) w_sum[warp] = make_uint4(ist, iac, ipd, wmax);
  __syncthreads();
  if (warp == 0) {
    uint4 v = lane < nwarps ? w_sum[lane] : make_uint4(0u, 0u, 0u, 0u);
    uint32_t x = v.x, y = v.y, z = v.z;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t a0 = __shfl_up_sync(kFullMask, x, off);
      const uint32_t a1 = __shfl_up_sync(kFullMask, y, off);
      const uint32_t a2 = __shfl_up_sync(kFullMask, z, off);
      if (lane >= off) {
        x += a0;
        y += a1;
        z += a2;
      }
    }
    const uint32_t m = __reduce_max_sync(kFullMask, v.w);
    w_sum[lane] = make_uint4(x - v.x, y - v.y, z - v.z, 0u);  // exclusive over warps
    if (lane == 31) s_total = make_uint4(x, y, z, m);
  }
  __syncthreads();
  const uint4 wb = w_sum[warp];
  uint32_t rst = wb.x + ist - st, rac = wb.y + iac - ac, rpd = wb.z + ipd - pd;
  for (int e = beg; e < end; ++e) {
    const uint32_t c = tot[e];
    start[e] = rst;
    act[e] = rac;
    pad[e] = rpd;
    rst += c;
    rac += c > 0u;
    rpd += (c + (kScaleRowAlign - 1)) / kScaleRowAlign * kScaleRowAlign;
  }
  const uint4 t = s_total;
  __syncthreads();
  TableSums r;
  r.slots = t.x;
  r.active = t.y;
  r.padded_total = t.z;
  r.max_count = t.w;
  return r;
}

// This CTA's share of the expert table (compact CSR, expert_ids, the
// optional scale offsets; CTA 0 also the usage stats). Thread g = b*blockDim
// + tid of the grid takes experts g, g + B*blockDim, ... and the tail
// entries A + g, ... (A active experts), so one CTA covers E <= blockDim.
__device__ void write_table_share(const IdxArgs& a, const uint32_t* tot, const uint32_t* start,
                                  const uint32_t* act, const uint32_t* pad, const TableSums& t) {
  const int E = a.E;
  const int stride = (int)(gridDim.x * blockDim.x);
  const int g0 = (int)(blockIdx.x * blockDim.x + threadIdx.x);
  for (int e = g0; e < E; e += stride) {
    if (tot[e] > 0u) {
      a.expert_ids[act[e]] = e;
      a.expert_start_indices[act[e]] = start[e];
      if (a.scales_offset) a.scales_offset[act[e]] = pad[e];
    }
  }
  const int A = (int)t.active;
  for (int j = A + g0; j <= E; j += stride) {
    a.expert_start_indices[j] = a.N;
    if (j < E) a.expert_ids[j] = -1;
    if (a.scales_offset) a.scales_offset[j] = t.padded_total;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.stats[0] = t.max_count;
    a.stats[1] = t.active;
  }
}

// Loads this warp's slots: -1 marks a slot past N or an id outside [0, E).
__device__ __forceinline__ void load_warp_slots(const IdxArgs& a, int64_t warp_base,
                                                int (&v)[kStepsPerWarp], bool& bad) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 0; s < kStepsPerWarp; ++s) {
    const int64_t i = warp_base + s * 32 + lane;
    int id = -1;
    if (i < (int64_t)a.N) {
      id = __ldcg(a.ids + i);
      if (id < 0 || id >= a.E) {
        bad = true;
        id = -1;
      }
    }
    v[s] = id;
  }
}

// ---------------------------------------------------------------- kernels shared by
// moe_create_indices and moe_route_index

// Where a scatter CTA takes its per-expert bases from.
enum BaseSource : int {
  kBasesSingleCta = 0,  // one CTA covers all slots: the bases are the expert starts
  kBasesFromCounts = 1  // the rows kernel turned the count matrix into prefixes
};

// One warp per expert e: exclusive prefix of the row counts[e][0..row) into
// prefix[e][..] (in place when they are the same array), 128 counts per pass
// (lane l takes counts 4l .. 4l+3 with one 16-byte load), and the row total to
// totals[e]. The padding columns are zero. With counts from the router the
// row is left zero for the next call's atomics, in the same coalesced pass.
__global__ void __launch_bounds__(kRowsWarps * 32) idx_rows_kernel(const IdxArgs a) {
  wait_for_prior_grid();
  // the status word starts here; the scatter CTAs add their bits to it (and
  // the count kernel's flags, when there is one)
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0u;
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRowsWarps + (threadIdx.x >> 5);
  if (e >= a.E) return;
  uint4* row = reinterpret_cast<uint4*>(a.counts + (int64_t)e * a.row);
  uint4* out = reinterpret_cast<uint4*>(a.prefix + (int64_t)e * a.row);
  const int Q = a.row / 4;
  uint32_t carry = 0;
  for (int q0 = 0; q0 < Q; q0 += 32) {
    const int q = q0 + lane;
    uint4 c = make_uint4(0u, 0u, 0u, 0u);
    if (q < Q) c = row[q];
    const uint32_t sum = c.x + c.y + c.z + c.w;
    uint32_t incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(kFullMask, incl, off);
      if (lane >= off) incl += y;
    }
    uint4 o;
    o.x = carry + incl - sum;
    o.y = o.x + c.x;
    o.z = o.y + c.y;
    o.w = o.z + c.z;
    if (q < Q) {
      out[q] = o;
      if (a.counts_from_router) row[q] = make_uint4(0u, 0u, 0u, 0u);
    }
    carry += __shfl_sync(kFullMask, incl, 31);
  }
  if (lane == 0) a.totals[e] = carry;
}


// Places CTA b's 1024 slots. Before the wait each warp ranks its slots: the
// rank of a slot is the number of earlier slots of its expert in the warp,
// found with one match per 32 slots while the previous kernel still runs.
// After it, base[e] = start of expert e + slots of e in earlier CTAs, the
// warps' running offsets follow from the per-warp counts, and each slot goes
// to base + running offset of its warp + its rank.
template <int kBases>
__global__ void __launch_bounds__(kIdxThreads) idx_scatter_kernel(const IdxArgs a) {
  extern __shared__ uint32_t smem[];
  uint32_t* s_warp = smem;                      // [kIdxWarps][E]
  uint32_t* s_base = s_warp + kIdxWarps * a.E;  // [E]
  uint32_t* s_act = s_base + a.E;               // [E]
  uint32_t* s_pad = s_act + a.E;                // [E]; then [E] totals, [E] prefixes
  // With the count matrix from the count and rows kernels, this kernel is the
  // third of the call, so the ids (written before the count kernel ran) are
  // complete once it starts: the ranking overlaps the rows kernel's tail.
  // A single CTA runs right after the ids' producer and must wait first.
  if constexpr (kBases == kBasesSingleCta) wait_for_prior_grid();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* my_cnt = s_warp + warp * a.E;
  for (int e = lane; e < a.E; e += 32) my_cnt[e] = 0;
  __syncwarp();

  const int64_t warp_base = (int64_t)blockIdx.x * kSlotsPerCta + warp * kSlotsPerWarp;
  int v[kStepsPerWarp];
  uint32_t rank[kStepsPerWarp];
  bool bad = false;
  load_warp_slots(a, warp_base, v, bad);
  const unsigned lower = lanemask_lt();
#pragma unroll
  for (int s = 0; s < kStepsPerWarp; ++s) {
    const unsigned peers = __match_any_sync(kFullMask, v[s]);
    rank[s] = v[s] >= 0 ? my_cnt[v[s]] + (uint32_t)__popc(peers & lower) : 0u;
    __syncwarp();
    if (v[s] >= 0 && lane == __ffs(peers) - 1) my_cnt[v[s]] += (uint32_t)__popc(peers);
    __syncwarp();
  }
  if constexpr (kBases == kBasesFromCounts) wait_for_prior_grid();  // counts, totals
  __syncthreads();

  const uint32_t* s_pre = nullptr;  // slots of each expert in earlier CTAs (null: none)
  bool consistent = true;
  if constexpr (kBases == kBasesSingleCta) {
    // the totals are the sums of the warps' counts; one blocked pass turns
    // them into the starts, active and padded offsets, and this CTA writes
    // the whole expert table
    uint32_t* s_tot = s_pad + a.E;  // [E]
    for (int e = threadIdx.x; e < a.E; e += kIdxThreads) {
      uint32_t t = 0;
      for (int w = 0; w < kIdxWarps; ++w) t += s_warp[w * a.E + e];
      s_tot[e] = t;
    }
    __syncthreads();
    const TableSums sums = scan_expert_table(s_tot, s_base, s_act, s_pad, a.E);
    write_table_share(a, s_tot, s_base, s_act, s_pad, sums);
    const int any_bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) *a.status = any_bad ? MOE_DEVICE_STATUS_BAD_EXPERT_ID : 0u;
  } else {
    // totals -> expert starts, active and padded offsets in one pass; every
    // CTA writes its share of the expert table, and CTA 0 ORs the count
    // kernel's flags (if any) into the status word the rows kernel zeroed
    __shared__ uint32_t s_flags;
    const int b = blockIdx.x;
    uint32_t* s_tot = s_pad + a.E;  // [E]
    uint32_t* pre = s_tot + a.E;    // [E]
    for (int e = threadIdx.x; e < a.E; e += kIdxThreads) {
      s_tot[e] = a.totals[e];
      pre[e] = a.prefix[(int64_t)e * a.row + b];
    }
    if (threadIdx.x == 0) s_flags = 0;
    __syncthreads();
    const TableSums sums = scan_expert_table(s_tot, s_base, s_act, s_pad, a.E);
    write_table_share(a, s_tot, s_base, s_act, s_pad, sums);
    s_pre = pre;
    // counts that do not add up to N can only come from a workspace that was
    // not zero-filled: reported, and no slot is placed (every position below
    // is also checked against N, so no write leaves the outputs)
    consistent = sums.slots == a.N;
    if (!consistent && b == 0 && threadIdx.x == 0) atomicOr(a.status, MOE_DEVICE_STATUS_SYNC_STATE);
    if (b == 0 && !a.counts_from_router) {
      uint32_t f = 0;
      for (int j = threadIdx.x; j < a.num_blocks; j += kIdxThreads) f |= a.flags[j];
      f = __reduce_or_sync(kFullMask, f);
      if (lane == 0 && f) atomicOr(&s_flags, f);
      __syncthreads();
      if (threadIdx.x == 0 && s_flags) atomicOr(a.status, s_flags);
    }
  }
  // per-warp running offsets: base + slots of e in earlier warps (the expert
  // table above only reads the starts, so no barrier is needed before this)
  for (int e = threadIdx.x; e < a.E; e += kIdxThreads) {
    uint32_t run = s_base[e] + (s_pre ? s_pre[e] : 0u);
    for (int w = 0; w < kIdxWarps; ++w) {
      const uint32_t c = s_warp[w * a.E + e];
      s_warp[w * a.E + e] = run;
      run += c;
    }
  }
  __syncthreads();

  bool overflow = false;
  if (consistent) {
#pragma unroll
    for (int s = 0; s < kStepsPerWarp; ++s) {
      const int64_t i = warp_base + s * 32 + lane;
      if (i < (int64_t)a.N) {
        const uint32_t pos = v[s] >= 0 ? my_cnt[v[s]] + rank[s] : 0xFFFFFFFFu;
        a.restore_token_order[i] = pos;
        if (v[s] >= 0) {
          if (pos < a.N)
            a.token_expert_order[pos] = (uint32_t)i;
          else
            overflow = true;
        }
      }
    }
  }
  if constexpr (kBases == kBasesFromCounts) {
    uint32_t bits = 0;
    if (a.counts_from_router && __any_sync(kFullMask, bad)) bits |= MOE_DEVICE_STATUS_BAD_EXPERT_ID;
    if (__any_sync(kFullMask, overflow)) bits |= MOE_DEVICE_STATUS_SYNC_STATE;
    if (bits && lane == 0) atomicOr(a.status, bits);
  }
}


}  // namespace
}  // namespace moe
