// Split-KV reduction (SparseAttnSharedkvMetadata, 参数说明, the `metadata`
// output, whose list also carries the per-core FlashDecode merge tasks),
// restated for one GPU. Each split s of a query tile left a normalised partial
// output O_s and its log-sum-exp lse_s; the merged row is
//   out = sum_s exp(lse_s - M) * O_s / sum_s exp(lse_s - M),  M = max_s lse_s.
// One warp merges 128 or 256 dims of one row; a CTA takes eight rows of one
// combine entry and one such slice (grid z).
#include <type_traits>

#include "pa_combine.cuh"
#include "pa_device.cuh"

namespace pa {

// DPL output dims a lane (4: 8-byte loads of the fp16 partials, 128 dims a
// warp; 8: 16-byte loads, 256 dims a warp, for value heads of 256 and more).
template <int DPL>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams C) {
  constexpr int kBatch = 16;  // splits whose partial rows a lane has in flight at once
  using Vec = typename std::conditional<DPL == 8, uint4, uint2>::type;  // DPL fp16 values
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (C.counts && int(blockIdx.x) >= C.counts[1]) return;
  // The work and combine lists were complete before the attention kernel
  // started: this entry and its first item are read while that kernel, whose
  // programmatic dependent this is, still runs.
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
  // the partial results: wait until the attention grid has finished and its
  // writes are visible
  grid_dependency_wait();
  const float* lse = C.part_lse + slot0 + rr;  // split s at lse[s * nrows]
  // this warp's 32 * DPL dims (blockIdx.z), DPL a lane; split s at po[s * split_stride]
  const int d = (blockIdx.z * 32 + lane) * DPL;
  const bool active = d < C.hv;
  const int64_t split_stride = int64_t(nrows) * C.hv;
  const __half* po = C.part_o + (int64_t(slot0) + rr) * C.hv + d;
  // The first batch of partial rows is loaded together with the LSEs: one
  // round trip to L2 before the arithmetic, not one per pass.
  Vec v[kBatch];
#pragma unroll
  for (int k = 0; k < kBatch; ++k)
    v[k] = (k < S && active) ? __ldg(reinterpret_cast<const Vec*>(po + k * split_stride)) : Vec{};
  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, __ldg(lse + int64_t(s) * nrows));
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float den = 0.f, w_lane = 0.f;  // lane s < 32 keeps split s's weight
  for (int s = lane; s < S; s += 32) {
    const float w = __expf(__ldg(lse + int64_t(s) * nrows) - M);
    if (s < 32) w_lane = w;
    den += w;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  float acc[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
  for (int s0 = 0; s0 < S; s0 += kBatch) {
    if (s0 > 0) {
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (s0 + k < S && active) v[k] = __ldg(reinterpret_cast<const Vec*>(po + (s0 + k) * split_stride));
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int s = s0 + k;
      if (s >= S) break;
      const float w = s < 32 ? __shfl_sync(0xffffffffu, w_lane, s)
                             : __expf(__ldg(lse + int64_t(s) * nrows) - M);
      const uint32_t* h = reinterpret_cast<const uint32_t*>(&v[k]);
#pragma unroll
      for (int j = 0; j < DPL / 2; ++j) {
        const float2 f = h2f2(h[j]);
        acc[2 * j] += w * f.x;
        acc[2 * j + 1] += w * f.y;
      }
    }
  }
  if (active) {
    const float inv = 1.f / den;
    const int r = r0 + rr, i = r / C.group, h = kvh * C.group + r % C.group;
    __half* dst = C.out + (int64_t(q_start + i) * C.num_heads + h) * C.hv;
    Vec pk;
    uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
    for (int j = 0; j < DPL / 2; ++j) pw[j] = pack_half2(acc[2 * j] * inv, acc[2 * j + 1] * inv);
    *reinterpret_cast<Vec*>(dst + d) = pk;
  }
}

cudaError_t launch_combine(const CombineParams& C, int64_t n_combine, int tile_rows,
                           cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  // 8 dims a lane (a 256-dim slice a warp) when the value head is a multiple of 256
  const bool wide = C.hv % 256 == 0;
  cfg.gridDim = dim3(unsigned(n_combine),
                     unsigned((tile_rows + kCombineThreads / 32 - 1) / (kCombineThreads / 32)),
                     unsigned(wide ? C.hv / 256 : (C.hv + 127) / 128));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return wide ? cudaLaunchKernelEx(&cfg, combine_kernel<8>, C)
              : cudaLaunchKernelEx(&cfg, combine_kernel<4>, C);
}

}  // namespace pa
