// Device helpers of libpa.so: shared-memory barriers, TMA copies and packed
// fp32 arithmetic for sm_103a, written as inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "pa.h"

namespace pa {

// A wait on an mbarrier gives up after this many SM clock cycles (about two
// seconds at GB300 clocks); a legitimate wait is microseconds. The decode
// kernels take the limit of their waits from FwdParams::wait_limit (this value
// unless a test lowers it); a wait for a CTA's own copies or tensor-core
// operations to finish before it exits (the drains and the teardown) always
// uses this one.
constexpr long long kWaitLimitCycles = 4ll << 30;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One poll of the phase with the given parity (the thread may be suspended
// inside it for a system-dependent time).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test without suspending the thread (returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete. Returns false
// when the wait ran out of time (more than `limit` SM clock cycles). Each poll
// (try_wait) may suspend the thread for a system-dependent time, so a limit
// far below that time does not make a wait run out: the wait returns as soon
// as its phase completes within the suspension.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// mbar_wait for the warp-pipelined kernels, whose waits are only on their own
// copies: under a lowered limit (tests) the polls do not suspend (test_wait),
// so that the limit, not the suspension, decides. The tcgen05 kernels keep
// mbar_wait: a second polling loop in their waits measured 7-10% slower, and
// their waits on other roles run out under a lowered limit as they are.
__device__ __forceinline__ bool mbar_wait_own(uint64_t* bar, uint32_t parity, long long limit) {
  if (limit < kWaitLimitCycles) {
    const long long t0 = clock64();
    while (!mbar_test_wait(bar, parity)) {
      if (clock64() - t0 > limit) return false;
    }
    return true;
  }
  return mbar_wait(bar, parity, limit);
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

// Prefetch one 2-D tensor-map box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// L2 policy for data read once per pass (the KV stream).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy for data that other CTAs read again soon (prefill K and V, read by
// every row tile of a sequence).
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Hardware base-2 exponential (MUFU.EX2); ex2(-inf) = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 fused multiply-add / multiply on register pairs (FFMA2/FMUL2 of
// sm_100 and later): d = a * b + c, lane-wise.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 h2f2(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2*>(&h);
  return __half22float2(v);
}

// Byte offset of a 16-byte chunk inside a TMA box written with a 32/64/128-byte
// swizzle: bits [4, 4+w) of the offset are XOR-ed with bits [7, 7+w).
__device__ __forceinline__ uint32_t swz(uint32_t off, uint32_t mask) {
  return off ^ (((off >> 7) & mask) << 4);
}

// Programmatic dependent launch: let the next kernel on the stream be
// scheduled (it still waits in grid_dependency_wait until this grid has
// completed and its memory operations are visible).
__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Maximum over the warp (redux.sync, float form of sm_100 and later).
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Sum over the warp.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Launch parameters shared by the attention kernels.
struct FwdParams {
  const __half* query;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* q_seqlens;  // may be null
  const __half* mask;        // may be null
  const float* alibi_slopes; // may be null
  const int32_t* work;
  const int32_t* counts;  // device plan: counts[0] items (CTAs past it exit), else null
  __half* out;
  uint32_t* status;
  __half* part_o;  // split items' rows, normalised, fp16
  float* part_lse;
  int64_t part_rows_cap;
  int num_heads, kv_heads, group, hk, hv, block_size, max_blocks_per_seq, num_blocks;
  int mask_type;
  int kv_shared;     // V of a token = the first hv dims of its K row (value_cache == key_cache)
  int q_tma;         // tcgen05 decode kernel: the query tile comes by TMA (tmq): 1 one box
                     // per 64-dim block, 2 one box for the tile (its rows are exactly G)
  int mask_q;        // PA_MASK_NORM: mask is [batch][mask_q][mask_kv]
  int64_t mask_kv;
  float scale_log2;  // scale * log2(e)
  long long wait_limit;  // cycles a wait on another role's progress may take
};

// Bias (base 2) of a PA_MASK_NORM mask for query token i of sequence b and key j.
__device__ __forceinline__ float norm_mask_log2(const FwdParams& P, int b, int i, int j) {
  return __half2float(P.mask[(int64_t(b) * P.mask_q + i) * P.mask_kv + j]) * kLog2e;
}

}  // namespace pa
