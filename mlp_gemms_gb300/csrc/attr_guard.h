// Per-device record of a kernel's launch attribute.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

namespace mx {

// Sets kernel K's dynamic shared-memory limit on the current device once.
// cudaFuncSetAttribute acts on the device the call is made on, so the record
// of which devices are done is kept per kernel and per device: a bitmask of
// device ordinals below 64, read and set atomically (threads may race to set
// it; setting it twice is harmless).  Ordinals past 63 set the attribute on
// every launch.
template <auto K>
cudaError_t ensure_smem_attr(int smem) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t)1 << dev : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace mx
