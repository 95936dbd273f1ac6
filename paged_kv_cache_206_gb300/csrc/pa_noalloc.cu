// pa_forward_noalloc: pa_forward with its workspace in a fixed device array
// owned by this library, for callers that must not allocate device memory.
//
// The workspace (status word, split-KV partial outputs and their log-sum-exps)
// lives in the file-scope array below, PA_NOALLOC_SCRATCH_BYTES large. Every
// GPU that loads the library holds that array until the process exits, and all
// calls on a device share it, so calls whose kernels overlap on the GPU (on
// different streams, or from different host threads) race with each other.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

// In host code this name is only a stand-in for the device array: its device
// address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_pa_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the array on the current device; looked up on the first
// call made with that device current, then cached.
pa_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_forward_noalloc(const pa_config* cfg, const void* query,
                                        const void* key_cache, const void* value_cache,
                                        const int32_t* block_tables, const int32_t* context_lens,
                                        const int32_t* q_seqlens, const void* mask,
                                        const float* alibi_slopes, const int32_t* work,
                                        int64_t n_items, const int32_t* combine,
                                        int64_t n_combine, size_t workspace_bytes,
                                        uint32_t* status, void* out, void* stream_) {
  if (workspace_bytes > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_BUFFER_TOO_SMALL;
  if (workspace_bytes < PA_STATUS_BYTES) workspace_bytes = PA_STATUS_BYTES;
  // pa_forward's own host checks first, so that a rejected call enqueues
  // nothing (the array is 256-byte aligned by its declaration)
  pa_status st = pa::check_forward(cfg, query, key_cache, value_cache, block_tables, context_lens,
                                   mask, alibi_slopes, work, n_items, combine, n_combine, nullptr,
                                   workspace_bytes, out, false);
  if (st != PA_OK) return st;
  void* scratch = nullptr;
  st = scratch_on_current_device(&scratch);
  if (st != PA_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  // The array keeps the previous call's contents: the status word must start at 0.
  // (Partial results are always written before they are read.)
  if (cudaMemsetAsync(scratch, 0, PA_STATUS_BYTES, stream) != cudaSuccess) return PA_ERR_CUDA;
  st = pa_forward(cfg, query, key_cache, value_cache, block_tables, context_lens, q_seqlens, mask,
                  alibi_slopes, work, n_items, combine, n_combine, scratch, workspace_bytes, out,
                  stream_);
  if (st != PA_OK) return st;
  if (status && cudaMemcpyAsync(status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                                stream) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}
