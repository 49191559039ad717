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
// column chunks (8 bf16) of the current token and issues all K row loads of
// several chunks (four per iteration in the 128-thread kernel) before the
// fp32 FMA chain, so every SM keeps many independent 16-byte loads in flight.
// Loads bypass L1 (each byte is used once), stores are streaming.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kFinThreads = 128;
// Chunks per thread and iteration: 4 in the 128-thread kernels (K = 2: 8
// loads of 16 bytes in flight per thread; K = 8: 32 loads, 164 registers,
// three CTAs per SM). Two chunks measured 7.5% slower with K = 2 (491 against
// 454 us, 131 072 tokens, H = 4096) and 1% slower with K = 8 (298.1 against
// 294.8 us, 16 384 tokens, H = 7168); six or eight were slower again. The
// wider CTAs of small batches keep 2 (at 512 threads 4 would spill).
constexpr int kChunkUnroll = 4;
constexpr int kChunkUnrollWide = 2;

struct FinArgs {
  void* out;           // [T, H] bf16 or fp32
  const uint4* down;   // [N, H8] 16-byte chunks of 8 bf16
  const uint32_t* restore;
  const void* weight;  // [T, K] fp32 or bf16
  int64_t T;
  int K;
  int64_t H8;  // hidden / 8
  uint32_t N;  // T * K
  uint32_t* status;  // optional: MOE_DEVICE_STATUS_BAD_RESTORE_ORDER for an entry >= N
};

// Records a skipped restore_order entry (one thread of the CTA reports it).
__device__ __forceinline__ void report_bad_restore(uint32_t* status) {
  if (status != nullptr) atomicOr(status, MOE_DEVICE_STATUS_BAD_RESTORE_ORDER);
}

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

// Router weight k of token t as fp32 (a bf16 weight widens exactly).
template <typename WT>
__device__ __forceinline__ float load_weight(const void* w, int64_t i) {
  if constexpr (sizeof(WT) == 4) {
    return __ldg(static_cast<const float*>(w) + i);
  } else {
    return __uint_as_float((uint32_t)__ldg(static_cast<const unsigned short*>(w) + i) << 16);
  }
}

// Chunk c (8 values) of output row t: bf16 rounded to nearest-even, or the fp32 sums.
template <typename OT>
__device__ __forceinline__ void store_chunk(void* out, int64_t t, int64_t H8, int64_t c,
                                            const float (&acc)[8]) {
  if constexpr (sizeof(OT) == 2) {
    uint32_t r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
      r[j] = *reinterpret_cast<uint32_t*>(&p);
    }
    __stcs(static_cast<uint4*>(out) + t * H8 + c, make_uint4(r[0], r[1], r[2], r[3]));
  } else {
    float4* o = static_cast<float4*>(out) + (t * H8 + c) * 2;
    __stcs(o, make_float4(acc[0], acc[1], acc[2], acc[3]));
    __stcs(o + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
  }
}

// K known at compile time: all K row loads of kUnroll chunks in flight.
// kThreads per CTA (one CTA per token): kFinThreads, or more for small
// batches so that a token's row takes fewer dependent rounds of loads.
template <int K, typename WT, typename OT, int kThreads = kFinThreads,
          int kUnroll = kChunkUnroll>
__global__ void __launch_bounds__(kThreads) finalize_kernel(const FinArgs a) {
  wait_for_prior_grid();
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    int64_t row[K];
    float w[K];
    bool ok[K];
    bool all_ok = true;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const uint32_t r = __ldg(a.restore + t * K + k);
      ok[k] = r < a.N;
      all_ok = all_ok && ok[k];
      row[k] = (int64_t)(ok[k] ? r : 0u) * a.H8;
      w[k] = load_weight<WT>(a.weight, t * K + k);
    }
    if (!all_ok && threadIdx.x == 0) report_bad_restore(a.status);
    for (int64_t c0 = threadIdx.x; c0 < a.H8; c0 += (int64_t)kThreads * kUnroll) {
      uint4 v[kUnroll][K];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = c0 + (int64_t)u * kThreads;
#pragma unroll
        for (int k = 0; k < K; ++k)
          v[u][k] = (c < a.H8 && ok[k]) ? load_stream(a.down + row[k] + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = c0 + (int64_t)u * kThreads;
        if (c >= a.H8) break;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < K; ++k) fma_bf16x8(acc, w[k], v[u][k]);
        store_chunk<OT>(a.out, t, a.H8, c, acc);
      }
    }
  }
}

// Any K <= 32: the rows go in blocks of kKBlock, all row loads of a block
// (kChunkUnroll chunks each) in flight before its FMAs, which keep k
// ascending. One row at a time (four loads in flight per thread) measured
// 393.4 us for K = 16 over 8192 tokens of H = 7168.
constexpr int kKBlock = 4;

template <typename WT, typename OT>
__global__ void __launch_bounds__(kFinThreads) finalize_kernel_any_k(const FinArgs a) {
  wait_for_prior_grid();
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    for (int64_t c0 = threadIdx.x; c0 < a.H8; c0 += (int64_t)kFinThreads * kChunkUnroll) {
      float acc[kChunkUnroll][8];
#pragma unroll
      for (int u = 0; u < kChunkUnroll; ++u)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[u][j] = 0.f;
      for (int kb = 0; kb < a.K; kb += kKBlock) {
        uint4 v[kKBlock][kChunkUnroll];
        float w[kKBlock];
        bool use[kKBlock];
#pragma unroll
        for (int j = 0; j < kKBlock; ++j) {
          const int k = kb + j;
          use[j] = k < a.K;
          const uint32_t r = use[j] ? __ldg(a.restore + t * a.K + k) : 0u;
          w[j] = use[j] ? load_weight<WT>(a.weight, t * a.K + k) : 0.0f;
          if (use[j] && r >= a.N) {
            if (threadIdx.x == 0 && c0 == 0) report_bad_restore(a.status);
            use[j] = false;
          }
          const uint4* src = a.down + (int64_t)(use[j] ? r : 0u) * a.H8;
#pragma unroll
          for (int u = 0; u < kChunkUnroll; ++u) {
            const int64_t c = c0 + (int64_t)u * kFinThreads;
            v[j][u] = (use[j] && c < a.H8) ? load_stream(src + c) : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int j = 0; j < kKBlock; ++j) {
          if (!use[j]) continue;
#pragma unroll
          for (int u = 0; u < kChunkUnroll; ++u) fma_bf16x8(acc[u], w[j], v[j][u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kChunkUnroll; ++u) {
        const int64_t c = c0 + (int64_t)u * kFinThreads;
        if (c < a.H8) store_chunk<OT>(a.out, t, a.H8, c, acc[u]);
      }
    }
  }
}

// One CTA per token: the block scheduler hands tokens to SMs as CTAs retire,
// so every SM streams until the last few tokens. A persistent grid of
// resident CTAs striding over the tokens ends unevenly (at 4 CTAs per SM and
// 16384 tokens some CTAs take 27 tokens, others 26) and measured about 1.3%
// slower. The token loop still strides, for T beyond the grid limit.
// A decode-sized batch (fewer tokens than four CTAs per SM) launches fully
// ordered after the index build: with programmatic serialisation a decode
// step (route + index + finalize, 128 tokens, replayed from a CUDA graph)
// measured 10.9 us against 10.3 us without it.
template <typename Kernel>
moe_status_t launch_fin(Kernel k, const FinArgs& a, cudaStream_t stream,
                        int threads = kFinThreads) {
  const int64_t cap = 0x7fffffff;
  const int grid = (int)(a.T < cap ? a.T : cap);
  if (a.T < 4 * (int64_t)device_info().sm_count)
    return launch_ordered(k, grid, threads, 0, stream, a);
  return launch(k, grid, threads, 0, stream, a);
}

// K fixed at compile time. When one round of loads at two chunks per thread
// needs more than kFinThreads threads, a batch with at most one token per SM
// takes up to 512 threads per token and one with at most two up to 256 (two
// chunks per thread; still one wave of CTAs at the registers a thread
// holds): a decode token's row of H = 7168 then takes one round, and a decode
// step (route + index + finalize, 128 tokens, replayed from a CUDA graph)
// measured 9.4 us against 10.2 us with 128 threads. Short rows and larger
// batches take the 128-thread kernel.
template <int K, typename WT, typename OT>
moe_status_t launch_fin_k(const FinArgs& a, cudaStream_t stream) {
  const int64_t sms = device_info().sm_count;
  const int64_t one_round = (a.H8 + kChunkUnrollWide - 1) / kChunkUnrollWide;  // threads
  if (one_round > 256 && a.T <= sms)
    return launch_fin(finalize_kernel<K, WT, OT, 512, kChunkUnrollWide>, a, stream, 512);
  if (one_round > kFinThreads && a.T <= 2 * sms)
    return launch_fin(finalize_kernel<K, WT, OT, 256, kChunkUnrollWide>, a, stream, 256);
  return launch_fin(finalize_kernel<K, WT, OT>, a, stream);
}

using bf16_t = unsigned short;

// fp32 weights, bf16 output: every specialised K.
moe_status_t dispatch_default(const FinArgs& a, cudaStream_t stream) {
  switch (a.K) {
    case 1: return launch_fin_k<1, float, bf16_t>(a, stream);
    case 2: return launch_fin_k<2, float, bf16_t>(a, stream);
    case 4: return launch_fin_k<4, float, bf16_t>(a, stream);
    case 6: return launch_fin_k<6, float, bf16_t>(a, stream);
    case 8: return launch_fin_k<8, float, bf16_t>(a, stream);
    default: return launch_fin(finalize_kernel_any_k<float, bf16_t>, a, stream);
  }
}

// Other dtype pairs: K = 2 and K = 8 specialised, the rest generic.
template <typename WT, typename OT>
moe_status_t dispatch_typed(const FinArgs& a, cudaStream_t stream) {
  switch (a.K) {
    case 2: return launch_fin_k<2, WT, OT>(a, stream);
    case 8: return launch_fin_k<8, WT, OT>(a, stream);
    default: return launch_fin(finalize_kernel_any_k<WT, OT>, a, stream);
  }
}

// Shared argument checks; fills `a` on success.
moe_status_t check_and_pack(void* output, size_t out_elem, const moe_bf16_t* down,
                            const uint32_t* restore_order, const void* router_weight,
                            size_t w_elem, int64_t T, int K, int64_t hidden, FinArgs* a) {
  if (T < 0 || K < 1 || hidden < 0) return MOE_ERR_INVALID_ARG;
  if (hidden % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (K > MOE_MAX_EXPERTS_PER_TOK) return MOE_ERR_UNSUPPORTED;
  if (T * (int64_t)K > (int64_t)0xFFFFFFFFu) return MOE_ERR_UNSUPPORTED;
  if (T == 0 || hidden == 0) return MOE_OK;
  if (!output || !down || !restore_order || !router_weight) return MOE_ERR_NULL_PTR;
  if (!aligned(output, 16) || !aligned(down, 16) || !aligned(restore_order, 4) ||
      !aligned(router_weight, w_elem))
    return MOE_ERR_MISALIGNED;
  // output must not overlap down (the kernel reads down while writing output)
  const uintptr_t o0 = (uintptr_t)output, o1 = o0 + (uintptr_t)(T * hidden * out_elem);
  const uintptr_t d0 = (uintptr_t)down, d1 = d0 + (uintptr_t)(T * K * hidden * 2);
  if (o0 < d1 && d0 < o1) return MOE_ERR_INVALID_ARG;
  a->out = output;
  a->down = reinterpret_cast<const uint4*>(down);
  a->restore = restore_order;
  a->weight = router_weight;
  a->T = T;
  a->K = K;
  a->H8 = hidden / 8;
  a->N = (uint32_t)(T * K);
  a->status = nullptr;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_finalize(moe_bf16_t* output, const moe_bf16_t* down,
                                     const uint32_t* restore_order, const float* router_weight,
                                     int64_t num_tokens, int32_t num_experts_per_token,
                                     int64_t hidden, cudaStream_t stream) {
  using namespace moe;
  FinArgs a{};
  const moe_status_t st = check_and_pack(output, 2, down, restore_order, router_weight, 4,
                                         num_tokens, num_experts_per_token, hidden, &a);
  if (st != MOE_OK || num_tokens == 0 || hidden == 0) return st;
  return dispatch_default(a, stream);
}

extern "C" moe_status_t moe_finalize_ex(void* output, moe_dtype_t output_dtype,
                                        const moe_bf16_t* down, const uint32_t* restore_order,
                                        const void* router_weight, moe_dtype_t weight_dtype,
                                        int64_t num_tokens, int32_t num_experts_per_token,
                                        int64_t hidden, uint32_t* device_status,
                                        cudaStream_t stream) {
  using namespace moe;
  const bool out_f32 = output_dtype == MOE_DTYPE_F32, w_f32 = weight_dtype == MOE_DTYPE_F32;
  if ((output_dtype != MOE_DTYPE_BF16 && !out_f32) || (weight_dtype != MOE_DTYPE_BF16 && !w_f32))
    return MOE_ERR_UNSUPPORTED;
  FinArgs a{};
  const moe_status_t st = check_and_pack(output, out_f32 ? 4 : 2, down, restore_order,
                                         router_weight, w_f32 ? 4 : 2, num_tokens,
                                         num_experts_per_token, hidden, &a);
  if (st != MOE_OK || num_tokens == 0 || hidden == 0) return st;
  if (!aligned(device_status, 4)) return MOE_ERR_MISALIGNED;
  a.status = device_status;
  if (w_f32 && !out_f32) return dispatch_default(a, stream);
  if (w_f32 && out_f32) return dispatch_typed<float, float>(a, stream);
  if (!w_f32 && !out_f32) return dispatch_typed<bf16_t, bf16_t>(a, stream);
  return dispatch_typed<bf16_t, float>(a, stream);
}
