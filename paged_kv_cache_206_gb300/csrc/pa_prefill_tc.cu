// Instantiations and launcher of the tcgen05 kernel for many-key tiles.
#include "pa_launch.h"
#include "pa_prefill_tc.cuh"

namespace pa {

cudaError_t launch_pf(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                      int64_t n_items, cudaStream_t stream) {
  auto go = [&](auto kern, uint32_t bytes) -> cudaError_t {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), int(bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(n_items), kPfThreads, bytes, stream>>>(tmk, tmv, P);
    return cudaGetLastError();
  };
  switch (P.hk) {
    case 64: return go(pf_attn_kernel<64>, PfCfg<64>::bytes);
    case 128: return go(pf_attn_kernel<128>, PfCfg<128>::bytes);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
