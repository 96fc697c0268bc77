// Host-side launch helpers shared by the kernels' launchers.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace mla {

// Raise a kernel's dynamic shared-memory limit on the current device, once
// per device: the attribute belongs to the kernel's instance on one device,
// so a process with contexts on several GPUs needs it on each.  `done` is
// the call site's record (bit d = device d; devices beyond 63 are set on
// every call).
template <class Kernel>
inline cudaError_t smem_attr_once(std::atomic<uint64_t>& done, Kernel kern, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace mla
