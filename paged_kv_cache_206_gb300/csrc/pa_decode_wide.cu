// Instantiations and launcher of the 16-row warp-level MMA decode kernel.
#include "pa_decode_wide.cuh"
#include "pa_launch.h"

namespace pa {

cudaError_t launch_wide(const CUtensorMap& tmk, const FwdParams& P, int64_t n_items,
                        cudaStream_t stream) {
  auto go = [&](auto kern, uint32_t bytes) -> cudaError_t {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), int(bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(n_items), kWideThreads, bytes, stream>>>(tmk, P);
    return cudaGetLastError();
  };
  switch (P.hk * 1000 + P.hv) {
    case 256256: return go(wide_decode_kernel<256, 256>, WideCfg<256, 256>::bytes);
    case 512512: return go(wide_decode_kernel<512, 512>, WideCfg<512, 512>::bytes);
    case 576512: return go(wide_decode_kernel<576, 512>, WideCfg<576, 512>::bytes);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
