// Launcher of the two-SM prefill kernel: one cluster of two CTAs per work item.
#include "pa_launch.h"
#include "pa_prefill_duo.cuh"

namespace pa {

cudaError_t launch_pf_duo(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                          int64_t n_items, cudaStream_t stream) {
  if (P.hk != 128 || P.hv != 128) return cudaErrorInvalidValue;
  const void* kern = reinterpret_cast<const void*>(pf_duo_kernel);
  cudaError_t e = ensure_smem_attr(kern, int(DuoCfg::bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(2 * n_items));
  cfg.blockDim = dim3(kDuoThreads);
  cfg.dynamicSmemBytes = DuoCfg::bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pf_duo_kernel, tmk, tmv, P);
}

}  // namespace pa
