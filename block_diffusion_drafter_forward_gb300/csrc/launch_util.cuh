// Host-side launch helpers shared by the projection GEMM and attention launchers.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

namespace dflash {

// Raise kernel `kern`'s dynamic shared-memory limit to `bytes` on the current device, once per
// device.  A function attribute belongs to the device's context, so a process that drives
// several GPUs sets it on each; `done` holds one bit per device id below 64 (higher ids set
// it on every call, which is harmless).
template <typename K>
inline cudaError_t smem_attr_once(K kern, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace dflash
