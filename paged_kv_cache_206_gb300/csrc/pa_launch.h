// Host-side launch helpers shared by the kernel launchers of libpa.so.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <unordered_map>

namespace pa {

// Raise a kernel's dynamic shared-memory limit once per (kernel, device) rather
// than on every launch.
inline cudaError_t ensure_smem_attr(const void* kern, int bytes) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, int> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const uint64_t key = (reinterpret_cast<uint64_t>(kern) << 8) ^ uint64_t(dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
  }
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> lock(mu);
    int& v = done[key];
    if (v < bytes) v = bytes;
  }
  return e;
}

}  // namespace pa
