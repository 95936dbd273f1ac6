// pa_hbm_read_probe: a streaming read of a device buffer, the read-only
// ceiling the attention kernels (which read the KV cache and write little)
// are compared against.
#include <cuda_runtime.h>

#include "pa_probe.h"

namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeUnroll = 8;

// 32 bytes in one load (the 256-bit global load of sm_100 and later), L1
// bypassed, L2 evict-first; returns the XOR of its eight words.
struct alignas(32) Vec32 {
  uint32_t w[8];
};

__device__ __forceinline__ uint32_t ld_stream_xor(const Vec32* p) {
  uint32_t a, b, c, d, e, f, g, h;
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(a), "=r"(b), "=r"(c), "=r"(d), "=r"(e), "=r"(f), "=r"(g), "=r"(h)
      : "l"(p));
  return a ^ b ^ c ^ d ^ e ^ f ^ g ^ h;
}

// Thread t of the grid reads vectors t, t + T, t + 2T, ... (T = all threads),
// kProbeUnroll of them per round, so that one load instruction of a warp
// covers 1024 contiguous bytes and every round keeps 8 loads in flight.
__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const Vec32* buf, size_t n,
                                                                   uint32_t* sink) {
  const size_t T = size_t(gridDim.x) * blockDim.x;
  size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + (kProbeUnroll - 1) * T < n; i += kProbeUnroll * T) {
    uint32_t v[kProbeUnroll];
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) v[u] = ld_stream_xor(buf + i + u * T);
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) acc ^= v[u];
  }
  for (; i < n; i += T) acc ^= ld_stream_xor(buf + i);
#pragma unroll
  for (int o = 16; o; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace

extern "C" pa_status pa_hbm_read_probe(const void* buf, size_t bytes, int ctas_per_sm,
                                       uint32_t* sink, void* stream) {
  if (!buf || !sink || bytes == 0 || bytes % 32 != 0 ||
      reinterpret_cast<uintptr_t>(buf) % 32 != 0 || ctas_per_sm < 1 || ctas_per_sm > 8)
    return PA_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  read_probe_kernel<<<unsigned(sms * ctas_per_sm), kProbeThreads, 0,
                      static_cast<cudaStream_t>(stream)>>>(static_cast<const Vec32*>(buf),
                                                          bytes / 32, sink);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
