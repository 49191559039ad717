// Shared device/host helpers of the sm_103a MoE routing kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_routing.h"

namespace moe {

constexpr unsigned kFullMask = 0xffffffffu;

// Order-preserving map of an fp32 value to uint32: a > b (IEEE, finite) iff
// key(a) > key(b) as unsigned. -0 is folded to +0 first so that the two
// zeros compare equal, as IEEE comparison does. Key 0 is below every
// non-NaN value and marks "no candidate".
__device__ __forceinline__ uint32_t ordered_key(float v) {
  uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Per-device properties looked up once.
struct DeviceInfo {
  int sm_count;
};
DeviceInfo device_info();

// Raises `kernel`'s dynamic shared-memory limit on the current device to at
// least `bytes`. The largest size set so far is remembered per kernel and
// device, so repeated launches of the same shape make no further runtime
// call. Callers skip it below the default limit.
moe_status_t set_dynamic_smem(const void* kernel, size_t bytes);

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline moe_status_t launch_status() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Every kernel of the library starts with this: with programmatic dependent
// launch the grid may begin while the previous kernel on the stream is still
// finishing, and this waits until that kernel has completed and its writes are
// visible. It then lets the next kernel on the stream be scheduled onto SMs
// that this grid frees, so that its launch overlaps this grid's tail; that
// kernel waits in turn before it reads anything. Because every kernel releases
// its dependents only after its own wait, a kernel that has started knows
// that every grid two or more launches back has completed. Without
// programmatic launch both instructions return at once.
__device__ __forceinline__ void wait_for_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` on `stream` with programmatic stream serialisation, so its
// launch overlaps the tail of the preceding kernel (which it then waits for in
// wait_for_prior_grid).
template <typename... KArgs, typename... Args>
moe_status_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                    cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return launch_status();
}

// Launches `kernel` fully ordered after the preceding work on `stream` (no
// programmatic serialisation; its wait_for_prior_grid returns at once).
template <typename... KArgs, typename... Args>
moe_status_t launch_ordered(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return launch_status();
}

}  // namespace moe
