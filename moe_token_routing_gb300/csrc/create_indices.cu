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
//             CTA 0 zeroes the device status word.
//   scatter : CTA b scans the totals into expert starts start(e) and writes
//             its share of the compact CSR, expert_ids and scale offsets (CTA
//             0 also the usage stats, and ORs the count flags into the status
//             word), reads its column of prefixes, and re-reads its
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

moe_status_t launch_index(const IdxArgs& a, const Layout& L, cudaStream_t stream) {
  const size_t scatter_smem = sizeof(uint32_t) * (size_t)(kIdxWarps + 5) * a.E;
  if (scatter_smem > 40 * 1024) {  // large E: opt in above the default 48 KB block limit
    const int bytes = (int)scatter_smem;
    if (set_dynamic_smem((const void*)idx_scatter_kernel<kBasesSingleCta>, bytes) != MOE_OK ||
        set_dynamic_smem((const void*)idx_scatter_kernel<kBasesFromCounts>, bytes) != MOE_OK)
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
  IdxArgs a{};
  a.ids = topk_ids;
  a.token_expert_order = token_expert_order;
  a.expert_start_indices = expert_start_indices;
  a.restore_token_order = restore_token_order;
  a.expert_ids = expert_ids;
  a.stats = expert_usage_stats;
  a.scales_offset = scales_offset_p;
  a.counts_from_router = 0;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.totals = reinterpret_cast<uint32_t*>(ws + L.totals_off);
  a.flags = reinterpret_cast<uint32_t*>(ws + L.flags_off);
  a.counts = reinterpret_cast<uint32_t*>(ws + L.counts_off);
  a.prefix = a.counts;  // prefixes in place of the counts
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
  return *host_status == 0u ? MOE_OK : MOE_ERR_DEVICE_DATA;
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
  IdxArgs a{};
  a.ids = topk_ids;
  a.token_expert_order = token_expert_order;
  a.expert_start_indices = expert_start_indices;
  a.restore_token_order = restore_token_order;
  a.expert_ids = expert_ids;
  a.stats = expert_usage_stats;
  a.scales_offset = nullptr;
  a.counts_from_router = 0;
  a.status = device_status ? device_status : reinterpret_cast<uint32_t*>(ws);
  a.totals = reinterpret_cast<uint32_t*>(ws + L.totals_off);
  a.flags = reinterpret_cast<uint32_t*>(ws + L.flags_off);
  a.counts = reinterpret_cast<uint32_t*>(ws + L.counts_off);
  a.prefix = a.counts;  // prefixes in place of the counts
  a.N = (uint32_t)N;
  a.E = E;
  a.num_blocks = (int)(L.num_blocks > 0 ? L.num_blocks : 1);
  a.row = (int)L.row;
  return launch_index(a, L, stream);
}
