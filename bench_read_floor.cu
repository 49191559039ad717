// A launch that only reads: the per-launch floor, on this GPU, of a kernel
// that must read a buffer once and do nothing else with it. bench.py times it
// on the router's input bytes, so that the router's back-to-back figure can
// be read against what any single launch over the same bytes costs. It is a
// measurement aid built beside the bench, not part of the routing library.
//
// Each thread streams 16-byte words at a grid stride, four loads in flight
// per step, and adds them up; each CTA writes the sum of its threads to
// partial[blockIdx.x], so the caller can check that every word was read.
#include <cuda_runtime.h>
#include <stddef.h>

namespace {

constexpr int kMaxThreads = 512;

__global__ void __launch_bounds__(kMaxThreads)
    stream_read_kernel(const float4* __restrict__ p, size_t n4, float* __restrict__ partial) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  float acc = 0.0f;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    const float4 a = __ldcs(p + i);
    const float4 b = __ldcs(p + i + stride);
    const float4 c = __ldcs(p + i + 2 * stride);
    const float4 d = __ldcs(p + i + 3 * stride);
    acc += ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w)) +
           ((c.x + c.y) + (c.z + c.w)) + ((d.x + d.y) + (d.z + d.w));
  }
  for (; i < n4; i += stride) {
    const float4 a = __ldcs(p + i);
    acc += (a.x + a.y) + (a.z + a.w);
  }
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  __shared__ float warp_sum[kMaxThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += warp_sum[w];
    partial[blockIdx.x] = s;
  }
}

}  // namespace

// p: n4 16-byte words on the device (16-byte aligned); partial: `grid` floats
// on the device. block is a multiple of 32, at most 512. Returns the CUDA
// error of the launch (0 on success); an invalid shape returns -1 unlaunched.
extern "C" int read_floor_launch(const void* p, size_t n4, float* partial, int grid, int block,
                                 cudaStream_t stream) {
  if (p == nullptr || partial == nullptr || grid < 1 || block < 32 || block > kMaxThreads ||
      block % 32 != 0 || (reinterpret_cast<size_t>(p) & 15) != 0)
    return -1;
  stream_read_kernel<<<grid, block, 0, stream>>>(static_cast<const float4*>(p), n4, partial);
  return (int)cudaGetLastError();
}
