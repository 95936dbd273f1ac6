// Instantiations and launcher of the tcgen05 decode kernel (64-row tiles).
#include "pa_decode_tc.cuh"
#include "pa_launch.h"

namespace pa {

cudaError_t launch_tc(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                      int64_t n_items, cudaStream_t stream) {
  const TcLayout lay = tc_layout(P.hk);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), int(lay.bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(n_items), kTcThreads, lay.bytes, stream>>>(tmk, tmv, P);
    return cudaGetLastError();
  };
  switch (P.hk * 1000 + P.hv) {
    case 128128: return go(tc_decode_kernel<128, 128>);
    case 256256: return go(tc_decode_kernel<256, 256>);
    case 512512: return go(tc_decode_kernel<512, 512>);
    case 576512: return go(tc_decode_kernel<576, 512>);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
