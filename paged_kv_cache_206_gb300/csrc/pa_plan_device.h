// Launch interface of the device-side planner (pa_plan_device.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace pa {

struct DevPlanParams {
  const int32_t* context_lens;
  const int32_t* q_seqlens;  // may be null (every q = 1)
  int32_t* work;
  int32_t* combine;
  int32_t* counts;   // [PA_PLAN_COUNTS]: items, combine entries, partial rows, error
  uint32_t* status;  // workspace status word
  int64_t work_cap, comb_cap;
  int batch, num_heads, kv_heads, group, block_size, max_blocks_per_seq, maxq, tr;
  int chunk_blocks, num_sms, hk, hv;
};

cudaError_t launch_plan(const DevPlanParams& D, cudaStream_t stream);

}  // namespace pa
