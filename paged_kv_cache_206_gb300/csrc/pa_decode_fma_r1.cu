// Instantiation of the CUDA-core decode kernel for row tiles of up to 1 rows.
#include "pa_decode_fma.cuh"

namespace pa {
template cudaError_t launch_fma<1>(const CUtensorMap&, const CUtensorMap&, const FwdParams&,
                                    int64_t, cudaStream_t);
}  // namespace pa
