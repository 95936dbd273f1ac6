// Instantiations of the tcgen05 decode kernel for 16-row tiles.
#include "pa_decode_tc.cuh"
#include "pa_launch.h"

namespace pa {

template <>
cudaError_t launch_tc_rows<16>(const CUtensorMap& tmk, const CUtensorMap& tmv,
                               const CUtensorMap& tmq, const FwdParams& P, int64_t n_items,
                               cudaStream_t stream) {
  return launch_tc_rows_impl<16>(tmk, tmv, tmq, P, n_items, stream, ensure_smem_attr);
}

}  // namespace pa
