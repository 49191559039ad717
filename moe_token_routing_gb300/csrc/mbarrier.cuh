// mbarrier and bulk-copy (cp.async.bulk) wrappers for sm_103a, with a
// bounded wait.
//
// A warp starts a global-to-shared bulk copy whose completion an mbarrier
// counts (arrive.expect_tx by the issuing thread, complete_tx by the copy
// engine), and its threads wait for the barrier's phase. Every wait is
// bounded: it gives up after one second of %globaltimer (or kSyncMaxPolls
// polls) and reports failure, so a copy that never completes ends in an
// error the caller handles, never in a hang.
#pragma once

#include <stdint.h>

#include "tagged_sync.cuh"

namespace moe {
namespace {

constexpr uint32_t kWaitHintNs = 1000000u;  // suspend-time hint of one mbarrier poll

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

// One poll of the phase with the given parity of `bar`; the thread may be
// suspended for up to kWaitHintNs while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kWaitHintNs)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity of `bar` has completed; false
// after one second of %globaltimer or kSyncMaxPolls polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t polls = 1; polls < kSyncMaxPolls; ++polls) {
    __nanosleep(64);
    if (mbar_try_wait(bar, parity)) return true;
    if ((polls & 31u) == 0u && global_ns() - t0 > kSyncTimeoutNs) return false;
  }
  return false;
}

}  // namespace
}  // namespace moe
