// Test harness (not part of the library): drives the bounded mbarrier wait of
// mbarrier.cuh, the wait the staged router uses for its score-chunk copies, on
// one CTA. With `complete`, thread 0 starts a 16-byte bulk copy that the
// barrier counts and the wait sees the phase complete; without it nothing
// ever arrives and the wait must give up on its own time limit. In both cases
// no copy is in flight when the kernel returns.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mbarrier.cuh"

namespace {

__global__ void mbar_selftest_kernel(const uint4* src, int complete, uint32_t* out,
                                     unsigned long long* elapsed_ns) {
  __shared__ __align__(16) uint4 dst;
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    moe::mbar_init(&bar, 1u);
    moe::fence_barrier_init();
    if (complete) {
      moe::mbar_arrive_expect_tx(&bar, sizeof(uint4));
      moe::bulk_copy_g2s(&dst, src, sizeof(uint4), &bar);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = moe::global_ns();
    const bool ok = moe::mbar_wait_bounded(&bar, 0u);
    *elapsed_ns = moe::global_ns() - t0;
    out[0] = ok ? 1u : 0u;
    out[1] = ok ? dst.x : 0u;
  }
}

}  // namespace

// src: 16 bytes of device memory; out: two device words (ok, first word
// copied); elapsed_ns: one device word. Returns the CUDA error of the launch
// and synchronisation.
extern "C" int mbar_wait_selftest(const void* src, int complete, uint32_t* out,
                                  unsigned long long* elapsed_ns) {
  mbar_selftest_kernel<<<1, 32>>>(static_cast<const uint4*>(src), complete, out, elapsed_ns);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return (int)e;
}
