// Library-wide pieces of the C ABI: status names and cached device facts.
#include <atomic>
#include <mutex>

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

moe_status_t set_dynamic_smem(const void* kernel, size_t bytes) {
  struct Entry {
    const void* kernel;
    int device;
    size_t bytes;
  };
  constexpr int kMaxEntries = 512;
  static Entry table[kMaxEntries];
  static int used = 0;
  static std::mutex lock;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> guard(lock);
  int slot = -1;
  for (int i = 0; i < used; ++i)
    if (table[i].kernel == kernel && table[i].device == dev) {
      if (table[i].bytes >= bytes) return MOE_OK;
      slot = i;
      break;
    }
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (slot < 0 && used < kMaxEntries) slot = used++;
  if (slot >= 0) table[slot] = Entry{kernel, dev, bytes};
  return MOE_OK;
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
    case MOE_ERR_DEVICE_DATA: return "MOE_ERR_DEVICE_DATA";
  }
  return "MOE_ERR_UNKNOWN";
}
