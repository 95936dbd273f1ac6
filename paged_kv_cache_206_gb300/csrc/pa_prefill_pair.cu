// Instantiations and launcher of the tcgen05 kernel for 256-row tiles.
#include "pa_launch.h"
#include "pa_prefill_pair.cuh"

namespace pa {

cudaError_t launch_pf_pair(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                           int64_t n_items, cudaStream_t stream) {
  auto go = [&](auto kern, uint32_t bytes) -> cudaError_t {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), int(bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(n_items), kPpThreads, bytes, stream>>>(tmk, tmv, P);
    return cudaGetLastError();
  };
  switch (P.hk) {
    case 64: return go(pf_pair_kernel<64>, PpCfg<64>::bytes);
    case 128: return go(pf_pair_kernel<128>, PpCfg<128>::bytes);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
