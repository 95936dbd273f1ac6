// Instantiations and launcher of the mma.sync decode kernel.
#include "pa_decode_mma.cuh"
#include "pa_launch.h"

namespace pa {

cudaError_t launch_mma(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                       int64_t n_items, cudaStream_t stream) {
  const int nw = mma_warps(P.hk, P.hv);
  const PipeLayout lay = pipe_layout(nw, kMmaBufs, P.hk, P.hv, 0, 8);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), int(lay.bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(n_items), nw * 32, lay.bytes, stream>>>(tmk, tmv, P);
    return cudaGetLastError();
  };
  if (P.hk == 64) return go(mma_decode_kernel<64, 64>);
  if (P.hk == 128) return go(mma_decode_kernel<128, 128>);
  if (P.hk == 256) return go(mma_decode_kernel<256, 256>);
  if (P.hk == 512) return go(mma_decode_kernel<512, 512>);
  return go(mma_decode_kernel<576, 512>);
}

}  // namespace pa
