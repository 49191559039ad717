// Expert-order permute of the token rows for sm_103a.
//
// Page "moe_create_indices", description paragraph: tokens are grouped by
// their assigned expert so that downstream kernels such as the grouped matmul
// can process each expert's tokens contiguously. This kernel builds that
// expert-contiguous input: row p of the output is the input row of the token
// that owns slot token_expert_order[p], i.e. output[restore_token_order[t*K+k]]
// = input[t] for every token t and k < K.
//
// HBM-bound, the mirror of finalize: each token row (2H bytes) is read once
// with 16-byte loads and written to its K destinations with streaming stores,
// so the bytes moved are 2*T*H + 2*T*K*H + 4*T*K.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kPermThreads = 128;
// Chunks per thread and iteration: 7 reads a 7168-wide row in one round at
// 128 threads. Against 2 (four rounds) it measured 323.5 against 326.7 us on
// the prefill workload (K = 8, H = 7168), the same on the few-expert one
// (K = 2, H = 4096: 469.4 us) and 94.1 against 94.3 us on the skewed one.
constexpr int kPermUnroll = 7;

struct PermArgs {
  uint4* out;        // [N, H8]
  const uint4* in;   // [T, H8]
  const uint32_t* restore;
  int64_t T;
  int K;
  int64_t H8;
  uint32_t N;
  uint32_t* status;  // optional: MOE_DEVICE_STATUS_BAD_RESTORE_ORDER for an entry >= N
};

__device__ __forceinline__ uint4 load_once(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int K>
__global__ void __launch_bounds__(kPermThreads) permute_kernel(const PermArgs a) {
  wait_for_prior_grid();
  const int k_count = K > 0 ? K : a.K;
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    int64_t dst[K > 0 ? K : 1];
    bool ok[K > 0 ? K : 1];
    if constexpr (K > 0) {
      bool all_ok = true;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const uint32_t r = __ldg(a.restore + t * K + k);
        ok[k] = r < a.N;
        all_ok = all_ok && ok[k];
        dst[k] = (int64_t)(ok[k] ? r : 0u) * a.H8;
      }
      if (!all_ok && threadIdx.x == 0 && a.status != nullptr)
        atomicOr(a.status, MOE_DEVICE_STATUS_BAD_RESTORE_ORDER);
    }
    const uint4* src = a.in + t * a.H8;
    for (int64_t c0 = threadIdx.x; c0 < a.H8; c0 += (int64_t)kPermThreads * kPermUnroll) {
      uint4 v[kPermUnroll];
#pragma unroll
      for (int u = 0; u < kPermUnroll; ++u) {
        const int64_t c = c0 + (int64_t)u * kPermThreads;
        v[u] = c < a.H8 ? load_once(src + c) : make_uint4(0, 0, 0, 0);
      }
      if constexpr (K > 0) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
          if (!ok[k]) continue;
#pragma unroll
          for (int u = 0; u < kPermUnroll; ++u) {
            const int64_t c = c0 + (int64_t)u * kPermThreads;
            if (c < a.H8) __stcs(a.out + dst[k] + c, v[u]);
          }
        }
      } else {
        for (int k = 0; k < k_count; ++k) {
          const uint32_t r = __ldg(a.restore + t * k_count + k);
          if (r >= a.N) {
            if (threadIdx.x == 0 && c0 == 0 && a.status != nullptr)
              atomicOr(a.status, MOE_DEVICE_STATUS_BAD_RESTORE_ORDER);
            continue;
          }
#pragma unroll
          for (int u = 0; u < kPermUnroll; ++u) {
            const int64_t c = c0 + (int64_t)u * kPermThreads;
            if (c < a.H8) __stcs(a.out + (int64_t)r * a.H8 + c, v[u]);
          }
        }
      }
    }
  }
}

template <int K>
moe_status_t launch_permute(const PermArgs& a, cudaStream_t stream) {
  // one CTA per token, as in finalize: tokens go to SMs as CTAs retire
  const int64_t cap = 0x7fffffff;
  const int grid = (int)(a.T < cap ? a.T : cap);
  return launch(permute_kernel<K>, grid, kPermThreads, 0, stream, a);
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute(moe_bf16_t* permuted, const moe_bf16_t* input,
                                    const uint32_t* restore_token_order, int64_t num_tokens,
                                    int32_t num_experts_per_token, int64_t hidden,
                                    uint32_t* device_status, cudaStream_t stream) {
  using namespace moe;
  const int64_t T = num_tokens;
  const int K = num_experts_per_token;
  if (T < 0 || K < 1 || hidden < 0) return MOE_ERR_INVALID_ARG;
  if (hidden % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (K > MOE_MAX_EXPERTS_PER_TOK) return MOE_ERR_UNSUPPORTED;
  if (T * (int64_t)K > (int64_t)0xFFFFFFFFu) return MOE_ERR_UNSUPPORTED;
  if (T == 0 || hidden == 0) return MOE_OK;
  if (!permuted || !input || !restore_token_order) return MOE_ERR_NULL_PTR;
  if (!aligned(permuted, 16) || !aligned(input, 16) || !aligned(restore_token_order, 4) ||
      !aligned(device_status, 4))
    return MOE_ERR_MISALIGNED;
  const uintptr_t o0 = (uintptr_t)permuted, o1 = o0 + (uintptr_t)(T * K * hidden * 2);
  const uintptr_t i0 = (uintptr_t)input, i1 = i0 + (uintptr_t)(T * hidden * 2);
  if (o0 < i1 && i0 < o1) return MOE_ERR_INVALID_ARG;

  PermArgs a{};
  a.out = reinterpret_cast<uint4*>(permuted);
  a.in = reinterpret_cast<const uint4*>(input);
  a.restore = restore_token_order;
  a.T = T;
  a.K = K;
  a.H8 = hidden / 8;
  a.N = (uint32_t)(T * K);
  a.status = device_status;
  switch (K) {
    case 1: return launch_permute<1>(a, stream);
    case 2: return launch_permute<2>(a, stream);
    case 4: return launch_permute<4>(a, stream);
    case 6: return launch_permute<6>(a, stream);
    case 8: return launch_permute<8>(a, stream);
    default: return launch_permute<0>(a, stream);
  }
}
