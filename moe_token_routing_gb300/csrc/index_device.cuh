// Device code of the expert index builder (page "moe_create_indices"),
// shared by the index kernels and the fused router + index kernel: the
// argument block, block-wide scans and the expert table (compact CSR,
// expert_ids, usage stats, aligned scale offsets).
#pragma once

#include "common.cuh"

namespace moe {
namespace {

constexpr int kIdxThreads = 256;
constexpr int kIdxWarps = kIdxThreads / 32;
constexpr int kStepsPerWarp = 4;
constexpr int kSlotsPerWarp = 32 * kStepsPerWarp;
constexpr int kSlotsPerCta = kIdxWarps * kSlotsPerWarp;  // 1024
constexpr int kScanThreads = 1024;
constexpr uint32_t kScaleRowAlign = MOE_SCALES_ROW_ALIGNMENT;

struct IdxArgs {
  const int32_t* ids;
  uint32_t* token_expert_order;
  uint32_t* expert_start_indices;
  uint32_t* restore_token_order;
  int32_t* expert_ids;
  uint32_t* stats;
  uint32_t* status;  // workspace word 0
  uint32_t* flags;   // [num_blocks]
  uint32_t* counts;  // [E][row]; the rows kernel turns each row into prefixes
  uint32_t* totals;  // [E]: slots of each expert
  uint32_t* scales_offset;  // optional [E+1]: 128-row aligned per-expert offsets
  uint32_t N;
  int E;
  int num_blocks;
  int row;
};

// ---------------------------------------------------------------- block helpers
// Exclusive prefix sum of data[0..n) in shared memory, in place; all threads of
// the block call it. Returns the total.
__device__ uint32_t block_exclusive_scan(uint32_t* data, int n, uint32_t* warp_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  const int per = (n + (int)blockDim.x - 1) / (int)blockDim.x;
  const int beg = min((int)threadIdx.x * per, n), end = min(beg + per, n);
  uint32_t local = 0;
  for (int i = beg; i < end; ++i) local += data[i];
  uint32_t x = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(kFullMask, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t v = lane < nwarps ? warp_tmp[lane] : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(kFullMask, v, off);
      if (lane >= off) v += y;
    }
    warp_tmp[lane] = v;
  }
  __syncthreads();
  uint32_t run = x - local + (warp > 0 ? warp_tmp[warp - 1] : 0u);
  const uint32_t total = warp_tmp[nwarps - 1];
  for (int i = beg; i < end; ++i) {
    const uint32_t v = data[i];
    data[i] = run;
    run += v;
  }
  __syncthreads();
  return total;
}

__device__ uint32_t block_max(uint32_t v, uint32_t* warp_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  v = __reduce_max_sync(kFullMask, v);
  if (lane == 0) warp_tmp[warp] = v;
  __syncthreads();
  uint32_t r = 0;
  for (int w = 0; w < nwarps; ++w) r = max(r, warp_tmp[w]);
  __syncthreads();
  return r;
}

// Given per-expert totals tot[0..E) in shared memory: writes the compact CSR,
// expert_ids and usage stats (and, if requested, the 128-row aligned scale
// offsets), and turns tot[] into each expert's start offset. `act` and `pad`
// are E words of shared scratch each.
__device__ void emit_expert_table(const IdxArgs& a, uint32_t* tot, uint32_t* act, uint32_t* pad,
                                  uint32_t* warp_tmp, bool write = true) {
  const bool want_scales = a.scales_offset != nullptr;
  uint32_t local_max = 0;
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    act[e] = tot[e] > 0u;
    if (want_scales) pad[e] = (tot[e] + (kScaleRowAlign - 1)) / kScaleRowAlign * kScaleRowAlign;
    local_max = max(local_max, tot[e]);
  }
  __syncthreads();
  const uint32_t max_count = block_max(local_max, warp_tmp);
  const uint32_t active = block_exclusive_scan(act, a.E, warp_tmp);
  block_exclusive_scan(tot, a.E, warp_tmp);  // tot[e] := start of expert e
  const uint32_t padded_total = want_scales ? block_exclusive_scan(pad, a.E, warp_tmp) : 0u;
  if (!write) return;
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    const bool is_active = (e + 1 < a.E ? act[e + 1] : active) != act[e];
    if (is_active) {
      a.expert_ids[act[e]] = e;
      a.expert_start_indices[act[e]] = tot[e];
      if (want_scales) a.scales_offset[act[e]] = pad[e];
    }
  }
  for (int j = (int)active + threadIdx.x; j <= a.E; j += blockDim.x) {
    a.expert_start_indices[j] = a.N;
    if (j < a.E) a.expert_ids[j] = -1;
    if (want_scales) a.scales_offset[j] = padded_total;
  }
  if (threadIdx.x == 0) {
    a.stats[0] = max_count;
    a.stats[1] = active;
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

}  // namespace
}  // namespace moe
