// Library-wide pieces of the C ABI: status names and cached device facts.
#include <atomic>

#include "common.cuh"

namespace moe {

DeviceInfo device_info() {
  constexpr int kMaxDevices = 64;
  static DeviceInfo cache[kMaxDevices];
  static std::atomic<bool> known[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    DeviceInfo d;
    d.sm_count = 1;
    return d;
  }
  if (!known[dev].load(std::memory_order_acquire)) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
    cache[dev].sm_count = n;
    known[dev].store(true, std::memory_order_release);
  }
  return cache[dev];
}

}  // namespace moe

extern "C" const char* moe_status_string(moe_status_t status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_NULL_PTR: return "MOE_ERR_NULL_PTR";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
  }
  return "MOE_ERR_UNKNOWN";
}
