// Fused unpermute gather + top-k weighted row sum for sm_103a.
//
// Page "moe_finalize", description paragraph: each output element reads its
// token's num_experts_per_token rows of down through restore_order, scales
// them by the router weights and accumulates in fp32, so the unpermuted
// [T, K, H] tensor never exists (Args output, down, restore_order,
// router_weight).
//
// HBM-bound: per token it streams K rows of 2H bytes from scattered
// positions of `down` and writes one 2H-byte row. Each thread owns 16-byte
// column chunks (8 bf16) of the current token and issues all K row loads of a
// chunk (two chunks per iteration) before the fp32 FMA chain, so every SM
// keeps many independent 16-byte loads in flight. Loads bypass L1 (each byte
// is used once), stores are streaming.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kFinThreads = 128;
constexpr int kChunkUnroll = 2;

struct FinArgs {
  uint4* out;          // [T, H8] 16-byte chunks
  const uint4* down;   // [N, H8]
  const uint32_t* restore;
  const float* weight;
  int64_t T;
  int K;
  int64_t H8;  // hidden / 8
  uint32_t N;  // T * K
};

__device__ __forceinline__ uint4 load_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float w, const uint4& v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    acc[2 * j] = __fmaf_rn(w, __uint_as_float(u[j] << 16), acc[2 * j]);
    acc[2 * j + 1] = __fmaf_rn(w, __uint_as_float(u[j] & 0xffff0000u), acc[2 * j + 1]);
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8]) {
  uint32_t r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    r[j] = *reinterpret_cast<uint32_t*>(&p);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// K known at compile time: all K row loads of kChunkUnroll chunks in flight.
template <int K>
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const FinArgs a) {
  wait_for_prior_grid();
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    int64_t row[K];
    float w[K];
    bool ok[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const uint32_t r = __ldg(a.restore + t * K + k);
      ok[k] = r < a.N;
      row[k] = (int64_t)(ok[k] ? r : 0u) * a.H8;
      w[k] = __ldg(a.weight + t * K + k);
    }
    uint4* out_row = a.out + t * a.H8;
    for (int64_t c0 = threadIdx.x; c0 < a.H8; c0 += (int64_t)kFinThreads * kChunkUnroll) {
      uint4 v[kChunkUnroll][K];
#pragma unroll
      for (int u = 0; u < kChunkUnroll; ++u) {
        const int64_t c = c0 + (int64_t)u * kFinThreads;
#pragma unroll
        for (int k = 0; k < K; ++k)
          v[u][k] = (c < a.H8 && ok[k]) ? load_stream(a.down + row[k] + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kChunkUnroll; ++u) {
        const int64_t c = c0 + (int64_t)u * kFinThreads;
        if (c >= a.H8) break;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < K; ++k) fma_bf16x8(acc, w[k], v[u][k]);
        __stcs(out_row + c, pack_bf16x8(acc));
      }
    }
  }
}

// Any K <= 32: one row load per step, chunks unrolled for some overlap.
__global__ void __launch_bounds__(kFinThreads) finalize_kernel_any_k(const FinArgs a) {
  wait_for_prior_grid();
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    uint4* out_row = a.out + t * a.H8;
    for (int64_t c0 = threadIdx.x; c0 < a.H8; c0 += (int64_t)kFinThreads * kChunkUnroll) {
      float acc[kChunkUnroll][8];
#pragma unroll
      for (int u = 0; u < kChunkUnroll; ++u)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[u][j] = 0.f;
      for (int k = 0; k < a.K; ++k) {
        const uint32_t r = __ldg(a.restore + t * a.K + k);
        const float w = __ldg(a.weight + t * a.K + k);
        if (r >= a.N) continue;
        const uint4* src = a.down + (int64_t)r * a.H8;
        uint4 v[kChunkUnroll];
#pragma unroll
        for (int u = 0; u < kChunkUnroll; ++u) {
          const int64_t c = c0 + (int64_t)u * kFinThreads;
          v[u] = c < a.H8 ? load_stream(src + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kChunkUnroll; ++u) fma_bf16x8(acc[u], w, v[u]);
      }
#pragma unroll
      for (int u = 0; u < kChunkUnroll; ++u) {
        const int64_t c = c0 + (int64_t)u * kFinThreads;
        if (c < a.H8) __stcs(out_row + c, pack_bf16x8(acc[u]));
      }
    }
  }
}

template <typename Kernel>
moe_status_t launch_fin(Kernel k, const FinArgs& a, cudaStream_t stream) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kFinThreads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t cap = (int64_t)device_info().sm_count * per_sm;
  const int grid = (int)(a.T < cap ? a.T : cap);
  return launch(k, grid, kFinThreads, 0, stream, a);
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_finalize(moe_bf16_t* output, const moe_bf16_t* down,
                                     const uint32_t* restore_order, const float* router_weight,
                                     int64_t num_tokens, int32_t num_experts_per_token,
                                     int64_t hidden, cudaStream_t stream) {
  using namespace moe;
  const int64_t T = num_tokens;
  const int K = num_experts_per_token;
  if (T < 0 || K < 1 || hidden < 0) return MOE_ERR_INVALID_ARG;
  if (hidden % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (K > MOE_MAX_EXPERTS_PER_TOK) return MOE_ERR_UNSUPPORTED;
  if (T * (int64_t)K > (int64_t)0xFFFFFFFFu) return MOE_ERR_UNSUPPORTED;
  if (T == 0 || hidden == 0) return MOE_OK;
  if (!output || !down || !restore_order || !router_weight) return MOE_ERR_NULL_PTR;
  if (!aligned(output, 16) || !aligned(down, 16) || !aligned(restore_order, 4) ||
      !aligned(router_weight, 4))
    return MOE_ERR_MISALIGNED;
  // output must not overlap down (the kernel reads down while writing output)
  const uintptr_t o0 = (uintptr_t)output, o1 = o0 + (uintptr_t)(T * hidden * 2);
  const uintptr_t d0 = (uintptr_t)down, d1 = d0 + (uintptr_t)(T * K * hidden * 2);
  if (o0 < d1 && d0 < o1) return MOE_ERR_INVALID_ARG;

  FinArgs a;
  a.out = reinterpret_cast<uint4*>(output);
  a.down = reinterpret_cast<const uint4*>(down);
  a.restore = restore_order;
  a.weight = router_weight;
  a.T = T;
  a.K = K;
  a.H8 = hidden / 8;
  a.N = (uint32_t)(T * K);
  switch (K) {
    case 1: return launch_fin(finalize_kernel<1>, a, stream);
    case 2: return launch_fin(finalize_kernel<2>, a, stream);
    case 4: return launch_fin(finalize_kernel<4>, a, stream);
    case 6: return launch_fin(finalize_kernel<6>, a, stream);
    case 8: return launch_fin(finalize_kernel<8>, a, stream);
    default: return launch_fin(finalize_kernel_any_k, a, stream);
  }
}
