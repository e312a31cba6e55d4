// launch_util.cuh -- host-side launch helpers shared by the kernel files.
#pragma once
#include <atomic>

#include <cuda_runtime.h>

namespace cg3 {

constexpr int kMaxDevices = 64;

// Dynamic shared memory above 48 KB needs a per-kernel, per-device attribute.  The attribute
// is raised only when a launch needs more than the value already set on the current device,
// so repeated launches make no attribute call.  `set_bytes` holds one entry per device.
template <class Kern>
cudaError_t ensure_dyn_smem(Kern* kernel, size_t smem, std::atomic<int>* set_bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices)
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (set_bytes[dev].load(std::memory_order_acquire) >= (int)smem) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int cur = set_bytes[dev].load(std::memory_order_relaxed);
  while (cur < (int)smem && !set_bytes[dev].compare_exchange_weak(cur, (int)smem)) {
  }
  return cudaSuccess;
}

}  // namespace cg3
