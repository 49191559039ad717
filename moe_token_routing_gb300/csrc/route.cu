// Group-limited top-k router for sm_103a.
//
// Page "group_limited_router_kernel", description paragraph: experts are split
// into n_groups groups, the topk_group best groups are kept and the
// n_experts_per_tok experts are chosen from them; the bias is added for the
// selection only (Args expert_bias, expert_weights); Parameters norm_weights
// and Args routed_scaling_factor fix the weight post-processing.
//
// Three kernel shapes:
//  * E = 32*L (L = 2 .. 32, a power of two), K <= 8, groups of whole lanes: L
//    lanes per token, 32 experts per lane; sorting networks over 32-bit
//    selection keys that carry the expert in their low bits, with the warp
//    path below as the exact fallback for near-equal scores (route_tokens_seg).
//  * other E > 32: one warp per token. Lane l holds the C = E/32 (rounded up to a
//    power of two) contiguous experts l*C .. l*C+C-1 in registers. Group
//    scores come from a per-lane top-2 plus a butterfly over the lanes of a
//    group; the expert top-K is K rounds of a warp-wide max (redux.sync on
//    order-preserving integer keys) where ties resolve to the lowest lane,
//    which holds the lowest expert index, because lanes hold ascending ranges.
//  * E <= 32: one thread per token, all E scores in registers.
// All three read each score row once with 16-byte (or scalar) loads, keep the bias
// in registers across a persistent token loop, and write K ids and weights
// per token.
#include "route_device.cuh"
#include "route_staged.cuh"

namespace moe {
namespace {

template <int C, bool kVec, bool kSoftmax>
__global__ void __launch_bounds__(kRouteThreads, C <= 8 ? 4 : 2) route_warp_kernel(const RouteArgs a) {
  extern __shared__ float dyn_smem[];  // kRouteWarps * a.warp_smem_words
  wait_for_prior_grid();
  const int warp = threadIdx.x >> 5;
  route_tokens_warp<C, kVec, kSoftmax>(a, (int64_t)blockIdx.x * kRouteWarps + warp, a.T,
                             (int64_t)gridDim.x * kRouteWarps, dyn_smem + warp * a.warp_smem_words,
                             [](int64_t, int, int) {});
}

template <int L, bool kGroups, bool kSoftmax>
__global__ void __launch_bounds__(kRouteThreads, 3) route_seg_kernel(const RouteArgs a) {
  extern __shared__ float dyn_smem[];  // softmax loader: a.warp_smem_words per warp
  __shared__ __align__(16) float s_bias[kSegBiasStride * (MOE_MAX_EXPERTS / kSegKeys)];
  __shared__ uint64_t s_cand[kRouteWarps * (32 / L) * kSegCand];
  __shared__ int s_slot[kRouteWarps * (32 / L) * kSegTop];
  wait_for_prior_grid();
  if (threadIdx.x < 32) stage_seg_bias(a, s_bias);
  __syncthreads();
  const int warps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5;
  route_tokens_seg<L, kGroups, kSoftmax>(a, s_bias, s_cand + warp * (32 / L) * kSegCand,
                               s_slot + warp * (32 / L) * kSegTop,
                               kSoftmax ? dyn_smem + warp * a.warp_smem_words : nullptr,
                               (int64_t)blockIdx.x * warps + warp,
                               (int64_t)gridDim.x * warps, [](int64_t, int, int) {});
}

// kKc: K fixed at compile time (8, the common case), or 0 for any K <= 8.
// kSigmoid / kSoftmax: the score loader (the softmax loader with K = 8 only).
template <int G, bool kSigmoid, int kKc, bool kSoftmax = false>
__global__ void __launch_bounds__(kStagedThreadsMax, 1) route_staged_kernel(const RouteArgs a,
                                                                           const StagedSplit sp) {
  extern __shared__ __align__(128) char staged_smem_buf[];
  wait_for_prior_grid();
  route_tokens_staged<kStagedR, G / kStagedR, kSigmoid, kKc, kSoftmax>(a, staged_smem_buf, sp,
                                                                        [](int64_t, int, int) {});
}

template <int EP, bool kVec>
__global__ void __launch_bounds__(kRouteThreads) route_thread_kernel(const RouteArgs a) {
  wait_for_prior_grid();
  route_tokens_thread<EP, kVec>(a, (int64_t)blockIdx.x * blockDim.x + threadIdx.x, a.T,
                                (int64_t)gridDim.x * blockDim.x, [](int64_t, int, int) {});
}

template <typename Kernel>
moe_status_t launch_route(Kernel k, const RouteArgs& a, int64_t tokens_per_cta, size_t smem,
                          cudaStream_t stream, int threads = kRouteThreads) {
  if (smem > 48 * 1024 && set_dynamic_smem((const void*)k, smem) != MOE_OK) return MOE_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (a.T + tokens_per_cta - 1) / tokens_per_cta;
  const int64_t cap = (int64_t)device_info().sm_count * per_sm;
  const int grid = (int)(want < cap ? want : cap);
  return launch(k, grid, threads, smem, stream, a);
}

template <int C, bool kSoftmax>
moe_status_t launch_warp_path_fn(const RoutePlan& p, cudaStream_t stream) {
  const size_t smem = route_warp_smem(p, kRouteWarps);
  if constexpr (C % 4 == 0) {
    if (p.vec)
      return launch_route(route_warp_kernel<C, true, kSoftmax>, p.a, kRouteWarps, smem, stream);
  }
  return launch_route(route_warp_kernel<C, false, kSoftmax>, p.a, kRouteWarps, smem, stream);
}

template <int C>
moe_status_t launch_warp_path(const RoutePlan& p, cudaStream_t stream) {
  if (p.a.score_fn == MOE_SCORES_SOFTMAX) return launch_warp_path_fn<C, true>(p, stream);
  return launch_warp_path_fn<C, false>(p, stream);
}

template <int L, bool kSoftmax>
moe_status_t launch_seg_path_fn(const RoutePlan& p, cudaStream_t stream) {
  const int warps = seg_warps_per_cta(p.a.T, L, device_info().sm_count);
  const int64_t tokens_per_cta = (int64_t)warps * (32 / L);
  const size_t smem = kSoftmax ? route_warp_smem(p, warps) : 0;
  if (p.a.group_mode == kGroupsAllKept)
    return launch_route(route_seg_kernel<L, false, kSoftmax>, p.a, tokens_per_cta, smem, stream,
                        32 * warps);
  return launch_route(route_seg_kernel<L, true, kSoftmax>, p.a, tokens_per_cta, smem, stream,
                      32 * warps);
}

template <int L>
moe_status_t launch_seg_path(const RoutePlan& p, cudaStream_t stream) {
  if (p.a.score_fn == MOE_SCORES_SOFTMAX) return launch_seg_path_fn<L, true>(p, stream);
  return launch_seg_path_fn<L, false>(p, stream);
}

template <int G, bool kSigmoid>
moe_status_t launch_staged_path_fn(const RoutePlan& p, cudaStream_t stream) {
  constexpr int kTok = 32 / kStagedR;
  if (p.a.K == kSegTop)
    return launch_staged(route_staged_kernel<G, kSigmoid, kSegTop>, p.a, p.a.T, p.a.E, kTok,
                         stream);
  return launch_staged(route_staged_kernel<G, kSigmoid, 0>, p.a, p.a.T, p.a.E, kTok, stream);
}

template <int G>
moe_status_t launch_staged_path(const RoutePlan& p, cudaStream_t stream) {
  constexpr int kTok = 32 / kStagedR;
  if (p.a.score_fn == MOE_SCORES_SOFTMAX)  // K = 8 (plan_route)
    return launch_staged(route_staged_kernel<G, false, kSegTop, true>, p.a, p.a.T, p.a.E, kTok,
                         stream);
  if (p.a.score_fn == MOE_SCORES_SIGMOID) return launch_staged_path_fn<G, true>(p, stream);
  return launch_staged_path_fn<G, false>(p, stream);
}

template <int EP>
moe_status_t launch_thread_path(const RoutePlan& p, cudaStream_t stream) {
  if (p.vec) return launch_route(route_thread_kernel<EP, true>, p.a, kRouteThreads, 0, stream);
  return launch_route(route_thread_kernel<EP, false>, p.a, kRouteThreads, 0, stream);
}

moe_status_t route_impl(int32_t* expert_indices, float* expert_weights,
                        const float* expert_scores, const float* expert_bias, int64_t num_tokens,
                        int32_t n_routed_experts, int32_t n_experts_per_tok, int32_t n_groups,
                        int32_t topk_group, int32_t norm_weights, float routed_scaling_factor,
                        int32_t score_fn, cudaStream_t stream) {
  RoutePlan p;
  moe_status_t st = plan_route(expert_indices, expert_weights, expert_scores, expert_bias,
                               num_tokens, n_routed_experts, n_experts_per_tok, n_groups,
                               topk_group, norm_weights, routed_scaling_factor, score_fn, &p);
  if (st != MOE_OK) return st;
  if (num_tokens == 0) return MOE_OK;
  st = check_route_pointers(p.a);
  if (st != MOE_OK) return st;
  switch (p.staged) {
    case 4: return launch_staged_path<4>(p, stream);
    case 8: return launch_staged_path<8>(p, stream);
    case 16: return launch_staged_path<16>(p, stream);
    default: break;
  }
  switch (p.seg) {
    case 2: return launch_seg_path<2>(p, stream);
    case 4: return launch_seg_path<4>(p, stream);
    case 8: return launch_seg_path<8>(p, stream);
    case 16: return launch_seg_path<16>(p, stream);
    case 32: return launch_seg_path<32>(p, stream);
    default: break;
  }
  switch (p.C) {
    case 0:
      if (p.EP == 8) return launch_thread_path<8>(p, stream);
      if (p.EP == 16) return launch_thread_path<16>(p, stream);
      return launch_thread_path<32>(p, stream);
    case 2: return launch_warp_path<2>(p, stream);
    case 4: return launch_warp_path<4>(p, stream);
    case 8: return launch_warp_path<8>(p, stream);
    case 16: return launch_warp_path<16>(p, stream);
    default: return launch_warp_path<32>(p, stream);
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route(int32_t* expert_indices, float* expert_weights,
                                  const float* expert_scores, const float* expert_bias,
                                  int64_t num_tokens, int32_t n_routed_experts,
                                  int32_t n_experts_per_tok, int32_t n_groups,
                                  int32_t topk_group, int32_t norm_weights,
                                  float routed_scaling_factor, cudaStream_t stream) {
  return moe::route_impl(expert_indices, expert_weights, expert_scores, expert_bias, num_tokens,
                         n_routed_experts, n_experts_per_tok, n_groups, topk_group, norm_weights,
                         routed_scaling_factor, MOE_SCORES_AS_GIVEN, stream);
}

extern "C" moe_status_t moe_route_ex(int32_t* expert_indices, float* expert_weights,
                                     const float* expert_scores, const float* expert_bias,
                                     int64_t num_tokens, int32_t n_routed_experts,
                                     int32_t n_experts_per_tok, int32_t n_groups,
                                     int32_t topk_group, int32_t norm_weights,
                                     float routed_scaling_factor, moe_score_fn_t score_fn,
                                     cudaStream_t stream) {
  return moe::route_impl(expert_indices, expert_weights, expert_scores, expert_bias, num_tokens,
                         n_routed_experts, n_experts_per_tok, n_groups, topk_group, norm_weights,
                         routed_scaling_factor, score_fn, stream);
}
