// Test harness (not part of the library): drives the bounded wait of
// tagged_sync.cuh on one CTA. Thread 0 waits for a tagged word; when asked,
// a thread of another warp of the same CTA publishes it after a short delay.
// Without a publisher the wait must give up on its own time limit.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tagged_sync.cuh"

namespace {

__global__ void selftest_kernel(uint64_t* word, uint32_t tag, int publish, uint32_t* out,
                                unsigned long long* elapsed_ns) {
  if (threadIdx.x == 32 && publish) {
    __nanosleep(20000);
    moe::store_tagged(word, tag, 1234u);
  }
  if (threadIdx.x == 0) {
    const uint64_t t0 = moe::global_ns();
    uint32_t v = 0;
    const bool ok = moe::wait_tagged(word, tag, v);
    *elapsed_ns = moe::global_ns() - t0;
    out[0] = ok ? 1u : 0u;
    out[1] = v;
  }
}

}  // namespace

// word: one 64-bit device word; out: two device words (ok, value); elapsed_ns:
// one device word. Returns the CUDA error of the launch and synchronisation.
extern "C" int tagged_sync_selftest(uint64_t* word, uint32_t tag, int publish, uint32_t* out,
                                    unsigned long long* elapsed_ns) {
  selftest_kernel<<<1, 64>>>(word, tag, publish, out, elapsed_ns);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return (int)e;
}
