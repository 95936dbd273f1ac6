// Launcher of the tcgen05 decode kernel, and its 64-row instantiations.
#include "pa_decode_tc.cuh"
#include "pa_launch.h"

namespace pa {

template <>
cudaError_t launch_tc_rows<64>(const CUtensorMap& tmk, const CUtensorMap& tmv,
                               const CUtensorMap& tmq, const FwdParams& P, int64_t n_items,
                               cudaStream_t stream) {
  return launch_tc_rows_impl<64>(tmk, tmv, tmq, P, n_items, stream, ensure_smem_attr);
}

cudaError_t launch_tc(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                      const FwdParams& P, int64_t n_items, cudaStream_t stream) {
  switch (tc_tile_rows(P.group, P.mask_q)) {
    case 16: return launch_tc_rows<16>(tmk, tmv, tmq, P, n_items, stream);
    case 32: return launch_tc_rows<32>(tmk, tmv, tmq, P, n_items, stream);
    default: return launch_tc_rows<64>(tmk, tmv, tmq, P, n_items, stream);
  }
}

}  // namespace pa
