// Expert index builder for sm_103a: a stable bucket sort of the flat router
// output by expert id.
//
// Page "moe_create_indices", description paragraph: slots are grouped by
// expert so that each expert's tokens are contiguous for the grouped matmul;
// Args token_expert_order, expert_start_indices, restore_token_order,
// expert_ids, expert_usage_stats, topk_ids. Parameters expected_count: the
// pages' kernel caches a bounded number of slots per expert in shared memory;
// here positions are computed arithmetically, so any count per expert works.
//
// Design (no inter-CTA waits, deterministic, stable):
//   count   : CTA b counts the experts of its 1024 slots, one per thread
//             (warp-aggregated with match.any, shared-memory counters) ->
//             counts[e][b] (expert-major, so one expert's counts are
//             contiguous).
//   rows    : one warp per expert turns its row into exclusive prefixes,
//             counts[e][b] := sum_{b' < b} counts[e][b'], and writes the total
//             tot[e]; each warp instruction covers 128 consecutive counts.
//   scatter : CTA b scans the totals into expert starts start(e) and writes
//             its share of the compact CSR, expert_ids and scale offsets (CTA
//             0 also the usage stats and the device status word), reads its
//             column of prefixes, and re-reads its
//             slots; within a CTA each warp owns 128 consecutive slots, so a
//             slot's position is start(e) + counts[e][b] + (slots of e in
//             earlier warps) + (slots of e in earlier steps of its warp) +
//             (lower lanes of its step with the same e). Writes
//             token_expert_order and restore_token_order in one pass.
//   For N <= 1024 one CTA does everything in one launch.
#include <mutex>

#include "index_device.cuh"

namespace moe {
namespace {

constexpr size_t kHeaderBytes = 256;
constexpr int kCountThreads = kSlotsPerCta;  // one slot per thread in the count kernel
constexpr int kRowsWarps = 8;                // rows kernel: warps per CTA, one expert each

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
  int64_t num_blocks;
  int64_t row;  // words per expert row of the count matrix (num_blocks rounded up to 4)
  size_t flags_off, counts_off, totals_off, total;
};

// Workspace: header (word 0: status) | flags [NB] | counts [E][row] | totals [E].
Layout workspace_layout(int64_t N, int E) {
  Layout L;
  L.num_blocks = (N + kSlotsPerCta - 1) / kSlotsPerCta;
  L.row = (L.num_blocks + 3) & ~(int64_t)3;
  L.flags_off = kHeaderBytes;
  if (L.num_blocks <= 1) {
    L.counts_off = L.totals_off = kHeaderBytes;
    L.total = kHeaderBytes;
  } else {
    L.counts_off = L.flags_off + align256(sizeof(uint32_t) * (size_t)L.num_blocks);
    L.totals_off = L.counts_off + align256(sizeof(uint32_t) * (size_t)L.row * (size_t)E);
    L.total = L.totals_off + align256(sizeof(uint32_t) * (size_t)E);
  }
  return L;
}

// ---------------------------------------------------------------- kernels
__global__ void __launch_bounds__(kCountThreads) idx_count_kernel(const IdxArgs a) {
  extern __shared__ uint32_t s_cnt[];  // [E]
  wait_for_prior_grid();
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t i = (int64_t)blockIdx.x * kSlotsPerCta + threadIdx.x;
  bool bad = false;
  int v = -1;
  if (i < (int64_t)a.N) {
    v = __ldg(a.ids + i);
    if (v < 0 || v >= a.E) {
      bad = true;
      v = -1;
    }
  }
  const unsigned peers = __match_any_sync(kFullMask, v);
  if (v >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_cnt[v], (uint32_t)__popc(peers));
  const int any_bad = __syncthreads_or(bad);
  for (int e = threadIdx.x; e < a.E; e += blockDim.x)
    a.counts[(int64_t)e * a.row + blockIdx.x] = s_cnt[e];
  if (blockIdx.x == a.num_blocks - 1) {  // padding columns of the count rows
    const int pad = a.row - a.num_blocks;
    for (int j = threadIdx.x; j < a.E * pad; j += blockDim.x)
      a.counts[(int64_t)(j / pad) * a.row + a.num_blocks + j % pad] = 0u;
  }
  if (threadIdx.x == 0) a.flags[blockIdx.x] = any_bad ? MOE_DEVICE_STATUS_BAD_EXPERT_ID : 0u;
}

// One warp per expert e: exclusive prefix of the row counts[e][0..row) in
// place, 128 counts per pass (lane l takes counts 4l .. 4l+3 with one 16-byte
// load), and the row total to totals[e]. The padding columns are zero.
__global__ void __launch_bounds__(kRowsWarps * 32) idx_rows_kernel(const IdxArgs a) {
  wait_for_prior_grid();
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRowsWarps + (threadIdx.x >> 5);
  if (e >= a.E) return;
  uint4* row = reinterpret_cast<uint4*>(a.counts + (int64_t)e * a.row);
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
    if (q < Q) row[q] = o;
    carry += __shfl_sync(kFullMask, incl, 31);
  }
  if (lane == 0) a.totals[e] = carry;
}

// Where a scatter CTA takes its per-expert bases from.
enum BaseSource : int {
  kBasesSingleCta = 0,  // one CTA covers all slots: the bases are the expert starts
  kBasesFromCounts = 1  // the last count CTA wrote them into the count matrix
};

template <int kBases>
__global__ void __launch_bounds__(kIdxThreads) idx_scatter_kernel(const IdxArgs a) {
  extern __shared__ uint32_t smem[];
  uint32_t* s_warp = smem;                      // [kIdxWarps][E]
  uint32_t* s_base = s_warp + kIdxWarps * a.E;  // [E]
  uint32_t* s_act = s_base + a.E;               // [E]
  uint32_t* s_pad = s_act + a.E;                // [E]; then [E] totals, [E] prefixes
  __shared__ uint32_t warp_tmp[32];
  // With the count matrix from the count and rows kernels, this kernel is the
  // third of the call, so the ids (written before the count kernel ran) are
  // complete once it starts: the warp counts overlap the rows kernel's tail.
  // A single CTA runs right after the ids' producer and must wait first.
  if constexpr (kBases == kBasesSingleCta) wait_for_prior_grid();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* my_cnt = s_warp + warp * a.E;
  for (int e = lane; e < a.E; e += 32) my_cnt[e] = 0;
  __syncwarp();

  const int64_t warp_base = (int64_t)blockIdx.x * kSlotsPerCta + warp * kSlotsPerWarp;
  int v[kStepsPerWarp];
  bool bad = false;
  load_warp_slots(a, warp_base, v, bad);

  // slots of each expert in this warp
#pragma unroll
  for (int s = 0; s < kStepsPerWarp; ++s) {
    const unsigned peers = __match_any_sync(kFullMask, v[s]);
    if (v[s] >= 0 && lane == __ffs(peers) - 1) my_cnt[v[s]] += (uint32_t)__popc(peers);
    __syncwarp();
  }
  if constexpr (kBases == kBasesFromCounts) wait_for_prior_grid();  // counts, totals
  __syncthreads();

  if constexpr (kBases == kBasesSingleCta) {
    for (int e = threadIdx.x; e < a.E; e += kIdxThreads) {
      uint32_t t = 0;
      for (int w = 0; w < kIdxWarps; ++w) t += s_warp[w * a.E + e];
      s_base[e] = t;
    }
    __syncthreads();
    emit_expert_table(a, s_base, s_act, s_pad, warp_tmp);
    const int any_bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) *a.status = any_bad ? MOE_DEVICE_STATUS_BAD_EXPERT_ID : 0u;
  } else {
    // totals -> expert starts, active and padded offsets in one pass; every
    // CTA writes its share of the expert table and CTA 0 the status word;
    // then base = start + this CTA's column of prefixes over earlier CTAs
    __shared__ uint32_t s_flags;
    const int b = blockIdx.x;
    uint32_t* s_tot = s_pad + a.E;  // [E]
    uint32_t* s_pre = s_tot + a.E;  // [E]
    for (int e = threadIdx.x; e < a.E; e += kIdxThreads) {
      s_tot[e] = a.totals[e];
      s_pre[e] = a.counts[(int64_t)e * a.row + b];
    }
    if (threadIdx.x == 0) s_flags = 0;
    __syncthreads();
    const TableSums sums = scan_expert_table(s_tot, s_base, s_act, s_pad, a.E);
    write_table_share(a, s_tot, s_base, s_act, s_pad, sums);
    for (int e = threadIdx.x; e < a.E; e += kIdxThreads) s_base[e] += s_pre[e];
    if (b == 0) {
      uint32_t f = 0;
      for (int j = threadIdx.x; j < a.num_blocks; j += kIdxThreads) f |= a.flags[j];
      f = __reduce_or_sync(kFullMask, f);
      if (lane == 0 && f) atomicOr(&s_flags, f);
      __syncthreads();
      if (threadIdx.x == 0) *a.status = s_flags;
    }
  }
  __syncthreads();
  // per-warp running offsets: base + slots of e in earlier warps
  for (int e = threadIdx.x; e < a.E; e += kIdxThreads) {
    uint32_t run = s_base[e];
    for (int w = 0; w < kIdxWarps; ++w) {
      const uint32_t c = s_warp[w * a.E + e];
      s_warp[w * a.E + e] = run;
      run += c;
    }
  }
  __syncthreads();

  const unsigned lower = lanemask_lt();
#pragma unroll
  for (int s = 0; s < kStepsPerWarp; ++s) {
    const int64_t i = warp_base + s * 32 + lane;
    const unsigned peers = __match_any_sync(kFullMask, v[s]);
    uint32_t pos = 0xFFFFFFFFu;
    if (v[s] >= 0) pos = my_cnt[v[s]] + (uint32_t)__popc(peers & lower);
    __syncwarp();
    if (v[s] >= 0 && lane == __ffs(peers) - 1) my_cnt[v[s]] += (uint32_t)__popc(peers);
    __syncwarp();
    if (i < (int64_t)a.N) {
      a.restore_token_order[i] = pos;
      if (v[s] >= 0) a.token_expert_order[pos] = (uint32_t)i;
    }
  }
}

moe_status_t launch_index(const IdxArgs& a, const Layout& L, cudaStream_t stream) {
  const size_t scatter_smem = sizeof(uint32_t) * (size_t)(kIdxWarps + 5) * a.E;
  if (scatter_smem > 40 * 1024) {  // large E: opt in above the default 48 KB block limit
    const int bytes = (int)scatter_smem;
    if (cudaFuncSetAttribute(idx_scatter_kernel<kBasesSingleCta>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(idx_scatter_kernel<kBasesFromCounts>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (L.num_blocks <= 1) {
    return launch(idx_scatter_kernel<kBasesSingleCta>, 1, kIdxThreads, scatter_smem, stream, a);
  }
  moe_status_t st =
      launch(idx_count_kernel, a.num_blocks, kCountThreads, sizeof(uint32_t) * a.E, stream, a);
  if (st != MOE_OK) return st;
  st = launch(idx_rows_kernel, (a.E + kRowsWarps - 1) / kRowsWarps, kRowsWarps * 32, 0, stream, a);
  if (st != MOE_OK) return st;
  return launch(idx_scatter_kernel<kBasesFromCounts>, a.num_blocks, kIdxThreads, scatter_smem,
                stream, a);
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_create_indices_workspace_size(int64_t num_slots, int32_t n_experts) {
  if (num_slots < 0 || n_experts < 1 || n_experts > MOE_MAX_EXPERTS) return 0;
  return moe::workspace_layout(num_slots, n_experts).total;
}

extern "C" moe_status_t moe_create_indices(uint32_t* token_expert_order,
                                           uint32_t* expert_start_indices,
                                           uint32_t* restore_token_order, int32_t* expert_ids,
                                           uint32_t* expert_usage_stats, const int32_t* topk_ids,
                                           int64_t num_slots, int32_t n_experts, void* workspace,
                                           size_t workspace_bytes, uint32_t* scales_offset_p,
                                           cudaStream_t stream) {
  using namespace moe;
  const int64_t N = num_slots;
  const int E = n_experts;
  if (N < 0 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > MOE_MAX_EXPERTS || N > (int64_t)0xFFFFFFFEu) return MOE_ERR_UNSUPPORTED;
  if (scales_offset_p != nullptr &&
      N + (int64_t)(kScaleRowAlign - 1) * E > (int64_t)0xFFFFFFFFu)
    return MOE_ERR_UNSUPPORTED;
  if (!expert_start_indices || !expert_ids || !expert_usage_stats) return MOE_ERR_NULL_PTR;
  if (N > 0 && (!token_expert_order || !restore_token_order || !topk_ids))
    return MOE_ERR_NULL_PTR;
  const Layout L = workspace_layout(N, E);
  if (!workspace || workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MOE_ERR_MISALIGNED;
  if (!aligned(token_expert_order, 4) || !aligned(expert_start_indices, 4) ||
      !aligned(restore_token_order, 4) || !aligned(expert_ids, 4) ||
      !aligned(expert_usage_stats, 4) || !aligned(topk_ids, 4) || !aligned(scales_offset_p, 4))
    return MOE_ERR_MISALIGNED;

  char* ws = static_cast<char*>(workspace);
  IdxArgs a;
  a.ids = topk_ids;
  a.token_expert_order = token_expert_order;
  a.expert_start_indices = expert_start_indices;
  a.restore_token_order = restore_token_order;
  a.expert_ids = expert_ids;
  a.stats = expert_usage_stats;
  a.scales_offset = scales_offset_p;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.totals = reinterpret_cast<uint32_t*>(ws + L.totals_off);
  a.flags = reinterpret_cast<uint32_t*>(ws + L.flags_off);
  a.counts = reinterpret_cast<uint32_t*>(ws + L.counts_off);
  a.N = (uint32_t)N;
  a.E = E;
  a.num_blocks = (int)(L.num_blocks > 0 ? L.num_blocks : 1);
  a.row = (int)L.row;
  return launch_index(a, L, stream);
}

extern "C" moe_status_t moe_read_device_status(const void* workspace, uint32_t* host_status,
                                               cudaStream_t stream) {
  if (!workspace || !host_status) return MOE_ERR_NULL_PTR;
  if (cudaMemcpyAsync(host_status, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

// ---------------------------------------------------------------- no-allocation variant
// Scratch of moe_create_indices_no_alloc: one array per device, created when
// the library is loaded and kept until the process exits. Host code may not
// use the name as an address (on the host it names a stand-in object); the
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[MOE_NO_ALLOC_SCRATCH_BYTES];

namespace moe {
namespace {

// Device address of g_no_alloc_scratch on the current device, looked up on
// the first call made on that device and cached.
moe_status_t no_alloc_scratch_address(void** out) {
  constexpr int kMaxDevices = 64;
  static void* addr[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_create_indices_no_alloc(uint32_t* token_expert_order,
                                                    uint32_t* expert_start_indices,
                                                    uint32_t* restore_token_order,
                                                    int32_t* expert_ids,
                                                    uint32_t* expert_usage_stats,
                                                    const int32_t* topk_ids, int64_t num_slots,
                                                    int32_t n_experts, uint32_t* device_status,
                                                    cudaStream_t stream) {
  using namespace moe;
  const int64_t N = num_slots;
  const int E = n_experts;
  if (N < 0 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > MOE_MAX_EXPERTS || N > (int64_t)0xFFFFFFFEu) return MOE_ERR_UNSUPPORTED;
  if (!expert_start_indices || !expert_ids || !expert_usage_stats) return MOE_ERR_NULL_PTR;
  if (N > 0 && (!token_expert_order || !restore_token_order || !topk_ids))
    return MOE_ERR_NULL_PTR;
  const Layout L = workspace_layout(N, E);
  if (L.total > (size_t)MOE_NO_ALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  if (!aligned(token_expert_order, 4) || !aligned(expert_start_indices, 4) ||
      !aligned(restore_token_order, 4) || !aligned(expert_ids, 4) ||
      !aligned(expert_usage_stats, 4) || !aligned(topk_ids, 4) || !aligned(device_status, 4))
    return MOE_ERR_MISALIGNED;

  void* scratch = nullptr;
  const moe_status_t st = no_alloc_scratch_address(&scratch);
  if (st != MOE_OK) return st;

  // Every scratch word that a kernel reads is written earlier in the same
  // call, so nothing has to be cleared between calls.
  char* ws = static_cast<char*>(scratch);
  IdxArgs a;
  a.ids = topk_ids;
  a.token_expert_order = token_expert_order;
  a.expert_start_indices = expert_start_indices;
  a.restore_token_order = restore_token_order;
  a.expert_ids = expert_ids;
  a.stats = expert_usage_stats;
  a.scales_offset = nullptr;
  a.status = device_status ? device_status : reinterpret_cast<uint32_t*>(ws);
  a.totals = reinterpret_cast<uint32_t*>(ws + L.totals_off);
  a.flags = reinterpret_cast<uint32_t*>(ws + L.flags_off);
  a.counts = reinterpret_cast<uint32_t*>(ws + L.counts_off);
  a.N = (uint32_t)N;
  a.E = E;
  a.num_blocks = (int)(L.num_blocks > 0 ? L.num_blocks : 1);
  a.row = (int)L.row;
  return launch_index(a, L, stream);
}
