// Launch interface of the split-KV reduction kernel.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "pa.h"

namespace pa {

constexpr int kCombineThreads = 256;     // 8 warps, one row each

struct CombineParams {
  const int32_t* combine;
  const int32_t* work;
  const __half* part_o;
  const float* part_lse;
  __half* out;
  uint32_t* status;
  int64_t part_rows_cap;
  int num_heads, group, hv;
  const int32_t* counts;  // device plan: counts[1] combine entries (CTAs past it exit), else null
};

cudaError_t launch_combine(const CombineParams& C, int64_t n_combine, int tile_rows,
                           cudaStream_t stream);

}  // namespace pa
