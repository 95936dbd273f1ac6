// Split-KV reduction: the FlashDecode reduction tasks of
// SparseAttnSharedkvMetadata (`metadata`: "每个vector核上FlashDecode的规约任务"),
// restated for one GPU. Each split s of a query tile left a normalised partial
// output O_s and its log-sum-exp lse_s; the merged row is
//   out = sum_s exp(lse_s - M) * O_s / sum_s exp(lse_s - M),  M = max_s lse_s.
// One warp merges 128 dims of one row; a CTA takes eight rows of one combine
// entry and one 128-dim slice (grid z).
#include "pa_combine.cuh"
#include "pa_device.cuh"

namespace pa {

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams C) {
  __shared__ float wts[kCombineThreads / 32][kCombineMaxSplits];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (C.counts && int(blockIdx.x) >= C.counts[1]) return;
  // Launched as a programmatic dependent of the attention kernel: wait until
  // that grid has finished and its partial results are visible.
  grid_dependency_wait();
  const int32_t* e = C.combine + int64_t(blockIdx.x) * PA_COMBINE_INTS;
  const int kvh = e[1], first = e[2], S = e[3];
  const int32_t* item = C.work + int64_t(first) * PA_WORK_INTS;
  const int r0 = item[2], r1 = item[3], q_start = item[6], slot0 = item[7];
  const int nrows = r1 - r0;
  if (slot0 < 0 || int64_t(slot0) + int64_t(S) * nrows > C.part_rows_cap) {
    if (threadIdx.x == 0) atomicOr(C.status, PA_STATUS_BIT_WORKSPACE);
    return;
  }
  const int rr = blockIdx.y * (kCombineThreads / 32) + warp;
  if (rr >= nrows) return;
  const float* lse = C.part_lse + slot0 + rr;  // split s at lse[s * nrows]
  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, lse[int64_t(s) * nrows]);
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float den = 0.f;
  for (int s = lane; s < S; s += 32) {
    const float w = __expf(lse[int64_t(s) * nrows] - M);
    if (s < kCombineMaxSplits) wts[warp][s] = w;
    den += w;
  }
  for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  __syncwarp();
  const float inv = 1.f / den;
  const int r = r0 + rr, i = r / C.group, h = kvh * C.group + r % C.group;
  __half* dst = C.out + (int64_t(q_start + i) * C.num_heads + h) * C.hv;
  const float* po = C.part_o + (int64_t(slot0) + rr) * C.hv;
  const int64_t split_stride = int64_t(nrows) * C.hv;
  // this warp's 128 dims (blockIdx.z); loads of several splits in flight at once
  const int d = blockIdx.z * 128 + lane * 4;
  if (d < C.hv) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int s = 0; s < S; ++s) {
      const float w = s < kCombineMaxSplits ? wts[warp][s] : __expf(lse[int64_t(s) * nrows] - M);
      const float4 v = __ldg(reinterpret_cast<const float4*>(po + s * split_stride + d));
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    __half2 lo = __floats2half2_rn(acc.x * inv, acc.y * inv);
    __half2 hi = __floats2half2_rn(acc.z * inv, acc.w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst + d) = pk;
  }
}

cudaError_t launch_combine(const CombineParams& C, int64_t n_combine, int tile_rows,
                           cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(n_combine),
                     unsigned((tile_rows + kCombineThreads / 32 - 1) / (kCombineThreads / 32)),
                     unsigned((C.hv + 127) / 128));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, C);
}

}  // namespace pa
