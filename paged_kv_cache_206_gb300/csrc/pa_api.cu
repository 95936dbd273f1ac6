// C ABI of libpa.so: argument checks, TMA descriptors and kernel launches.
// The operation and its constraints are those of PagedAttentionOperation
// ("Constraints"); the work list is built by pa_plan (pa_plan.cpp).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "pa.h"
#include "pa_testing.h"
#include "pa_combine.cuh"
#include "pa_decode_mma.cuh"
#include "pa_decode_wide.cuh"
#include "pa_decode_tc.cuh"
#include "pa_prefill_pair.cuh"
#include "pa_prefill_tc.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_plan_device.h"

namespace pa {

template <int RT>
cudaError_t launch_fma(const CUtensorMap&, const CUtensorMap&, const FwdParams&, int64_t,
                       cudaStream_t);

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct BoxGeom {
  int width;  // elements per row of one TMA box
  uint32_t swz_mask;
  CUtensorMapSwizzle swizzle;
};

// TMA box width and swizzle: 64-element (128-byte) boxes with the 128-byte
// swizzle when both head sizes are multiples of 64, else 16-element boxes
// with the 32-byte swizzle (16 divides every valid head size). Either way a
// column of 16-byte chunks read across consecutive token rows hits distinct
// shared-memory banks.
BoxGeom box_geom(bool wide) {
  if (wide) return {64, 7u, CU_TENSOR_MAP_SWIZZLE_128B};
  return {16, 1u, CU_TENSOR_MAP_SWIZZLE_32B};
}

// Encoded tensor maps of recent calls, keyed by everything the encoding reads,
// so that a steady stream of pa_forward calls on the same caches does not
// re-encode them.
struct MapKey {
  const void* base;
  uint64_t dims[3];
  uint32_t box[3];
  int rank, swizzle;
  bool operator==(const MapKey& o) const {
    return base == o.base && rank == o.rank && swizzle == o.swizzle && dims[0] == o.dims[0] &&
           dims[1] == o.dims[1] && dims[2] == o.dims[2] && box[0] == o.box[0] &&
           box[1] == o.box[1] && box[2] == o.box[2];
  }
};

class MapCache {
 public:
  bool get(const MapKey& k, CUtensorMap* out) {
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < kEntries; ++i)
      if (used_[i] && keys_[i] == k) {
        *out = maps_[i];
        return true;
      }
    return false;
  }
  void put(const MapKey& k, const CUtensorMap& m) {
    std::lock_guard<std::mutex> lock(mu_);
    keys_[next_] = k;
    maps_[next_] = m;
    used_[next_] = true;
    next_ = (next_ + 1) % kEntries;
  }

 private:
  static constexpr int kEntries = 16;
  std::mutex mu_;
  MapKey keys_[kEntries];
  CUtensorMap maps_[kEntries];
  bool used_[kEntries] = {};
  int next_ = 0;
};

MapCache& map_cache() {
  static MapCache c;
  return c;
}

// The map for key k (fp16 elements; the row stride follows from the dims).
bool cached_map(CUtensorMap* m, const MapKey& k, const cuuint64_t* strides) {
  if (map_cache().get(k, m)) return true;
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {k.dims[0], k.dims[1], k.dims[2]};
  cuuint32_t box[3] = {k.box[0], k.box[1], k.box[2]};
  cuuint32_t es[3] = {1, 1, 1};
  if (enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, cuuint32_t(k.rank), const_cast<void*>(k.base), dims,
          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CUtensorMapSwizzle(k.swizzle),
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  map_cache().put(k, *m);
  return true;
}

// The cache [num_blocks, bs, Hk, hs] viewed as a 2-D tensor of
// num_blocks * bs token rows by Hk * hs elements; a box is box_rows tokens of
// one box-width slice of one kv head.
bool cache_map(CUtensorMap* m, const void* base, const pa_config& c, int hs, int box_rows,
               const BoxGeom& g) {
  MapKey k{};
  k.base = base;
  k.rank = 2;
  k.swizzle = int(g.swizzle);
  k.dims[0] = uint64_t(c.kv_heads) * hs;
  k.dims[1] = uint64_t(c.num_blocks) * c.block_size;
  k.box[0] = uint32_t(g.width);
  k.box[1] = uint32_t(box_rows);
  const cuuint64_t strides[2] = {cuuint64_t(c.kv_heads) * hs * 2, 0};
  return cached_map(m, k, strides);
}

// The same cache as a 3-D tensor for the tcgen05 kernel: dims (64 elements of
// a head-dim block, token rows, head-dim blocks of all kv heads), strides
// (row stride, 128 bytes); a box is box_rows tokens x `halves` blocks of 64
// dims, each landing as its own [box_rows][128 B] swizzled tile.
bool cache_map_3d(CUtensorMap* m, const void* base, const pa_config& c, int hs, int box_rows,
                  int halves) {
  MapKey k{};
  k.base = base;
  k.rank = 3;
  k.swizzle = int(CU_TENSOR_MAP_SWIZZLE_128B);
  k.dims[0] = 64;
  k.dims[1] = uint64_t(c.num_blocks) * c.block_size;
  k.dims[2] = uint64_t(c.kv_heads) * (hs / 64);
  k.box[0] = 64;
  k.box[1] = uint32_t(box_rows);
  k.box[2] = uint32_t(halves);
  const cuuint64_t strides[2] = {cuuint64_t(c.kv_heads) * hs * 2, 128};
  return cached_map(m, k, strides);
}

// The query [batch, H, hk] of a launch with one query token per sequence, as a
// 3-D tensor for the tcgen05 kernel: dims (64 elements of a head-dim block,
// batch * H rows, hk / 64 blocks), strides (row stride hk * 2 bytes, 128); a
// box is G rows (the heads of one kv head, consecutive in memory) of
// `blocks_per_box` 64-dim blocks, landing as [block][G][128 B] with the
// 128-byte swizzle.
bool query_map(CUtensorMap* m, const void* query, const pa_config& c, int blocks_per_box) {
  MapKey k{};
  k.base = query;
  k.rank = 3;
  k.swizzle = int(CU_TENSOR_MAP_SWIZZLE_128B);
  k.dims[0] = 64;
  k.dims[1] = uint64_t(c.batch) * c.num_heads;
  k.dims[2] = uint64_t(c.head_size_k / 64);
  k.box[0] = 64;
  k.box[1] = uint32_t(c.num_heads / c.kv_heads);
  k.box[2] = uint32_t(blocks_per_box);
  const cuuint64_t strides[2] = {cuuint64_t(c.head_size_k) * 2, 128};
  return cached_map(m, k, strides);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Cycle limit of the decode kernels' waits on other roles (0: the default);
// set only through pa_testing_set_wait_limit.
std::atomic<long long> g_wait_limit{0};

}  // namespace

pa_status check_forward(const pa_config* cfg, const void* query, const void* key_cache,
                        const void* value_cache, const int32_t* block_tables,
                        const int32_t* context_lens, const void* mask, const float* alibi_slopes,
                        const int32_t* work, int64_t n_items, const int32_t* combine,
                        int64_t n_combine, const void* workspace, size_t workspace_bytes,
                        const void* out, bool check_workspace) {
  pa_status st = validate_config(cfg);
  if (st != PA_OK) return st;
  const pa_config& c = *cfg;
  if (!query || !key_cache || !value_cache || !block_tables || !context_lens || !out ||
      (check_workspace && !workspace))
    return PA_ERR_INVALID_ARG;
  const bool has_mask = c.mask_type == PA_MASK_NORM_COMPRESS || c.mask_type == PA_MASK_NORM;
  if (has_mask != (mask != nullptr)) return PA_ERR_INVALID_ARG;
  if ((c.mask_type == PA_MASK_ALIBI) != (alibi_slopes != nullptr)) return PA_ERR_INVALID_ARG;
  if (n_items < 0 || n_combine < 0 || n_items > INT32_MAX || n_combine > INT32_MAX)
    return PA_ERR_INVALID_ARG;
  if ((n_items > 0 && !work) || (n_combine > 0 && !combine)) return PA_ERR_INVALID_ARG;
  // value_cache == key_cache: the shared-KV layout, V = first hv dims of each K row
  if (value_cache == key_cache && c.head_size_v > c.head_size_k) return PA_ERR_INVALID_ARG;
  if (!aligned(query, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
      !aligned(out, 16) || (check_workspace && !aligned(workspace, 256)))
    return PA_ERR_INVALID_ARG;
  if (workspace_bytes < PA_STATUS_BYTES) return PA_ERR_BUFFER_TOO_SMALL;
  return PA_OK;
}

}  // namespace pa

namespace {

// The forward pass. With `counts` null the grids are n_items and n_combine
// CTAs; with a device plan they are the list capacities, and the CTAs past
// the device-side counts (counts[0] items, counts[1] combine entries) return
// at once.
pa_status forward_impl(const pa_config* cfg, const void* query, const void* key_cache,
                       const void* value_cache, const int32_t* block_tables,
                       const int32_t* context_lens, const int32_t* q_seqlens, const void* mask,
                       const float* alibi_slopes, const int32_t* work, int64_t n_items,
                       const int32_t* combine, int64_t n_combine, const int32_t* counts,
                       void* workspace, size_t workspace_bytes, void* out, void* stream_) {
  using namespace pa;
  const pa_status st = check_forward(cfg, query, key_cache, value_cache, block_tables,
                                     context_lens, mask, alibi_slopes, work, n_items, combine,
                                     n_combine, workspace, workspace_bytes, out, true);
  if (st != PA_OK) return st;
  const pa_config& c = *cfg;
  const bool kv_shared = value_cache == key_cache;
  if (n_items == 0) return PA_OK;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int64_t TR = tile_rows(c);
  const int hk = c.head_size_k, hv = c.head_size_v;
  const int64_t cap = workspace_rows(workspace_bytes, hv);
  const WorkspaceLayout wl = workspace_layout(cap, hv);

  FwdParams P{};
  P.query = static_cast<const __half*>(query);
  P.block_tables = block_tables;
  P.context_lens = context_lens;
  P.q_seqlens = q_seqlens;
  P.mask = static_cast<const __half*>(mask);
  P.alibi_slopes = alibi_slopes;
  P.work = work;
  P.out = static_cast<__half*>(out);
  P.status = static_cast<uint32_t*>(workspace);
  P.part_o = reinterpret_cast<__half*>(static_cast<char*>(workspace) + wl.partial_o);
  P.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + wl.partial_lse);
  P.part_rows_cap = cap;
  P.num_heads = c.num_heads;
  P.kv_heads = c.kv_heads;
  P.group = c.num_heads / c.kv_heads;
  P.hk = hk;
  P.hv = hv;
  P.block_size = c.block_size;
  P.max_blocks_per_seq = c.max_blocks_per_seq;
  P.num_blocks = c.num_blocks;
  P.mask_type = c.mask_type;
  P.kv_shared = kv_shared ? 1 : 0;
  P.counts = counts;
  P.mask_q = int(max_q(c));
  P.mask_kv = int64_t(c.max_blocks_per_seq) * c.block_size;
  const float scale = c.scale > 0.f ? c.scale : 1.0f / std::sqrt(float(hk));
  P.scale_log2 = scale * kLog2e;
  const long long wlim = g_wait_limit.load(std::memory_order_relaxed);
  P.wait_limit = wlim > 0 ? wlim : kWaitLimitCycles;

  cudaError_t err;
  if (TR <= PA_FMA_MAX_ROWS) {
    const bool wide = (hk % 64 == 0) && (hv % 64 == 0);
    CUtensorMap tmk, tmv;
    // (with a shared-KV cache the warp kernels read V from the K boxes; the
    // V map is then built over the K rows and left unused)
    if (wide) {
      // one 3-D box per 16-token sub-tile: every 64-dim block of the head
      if (!cache_map_3d(&tmk, key_cache, c, hk, 16, hk / 64) ||
          !cache_map_3d(&tmv, value_cache, c, kv_shared ? hk : hv, 16, hv / 64))
        return PA_ERR_CUDA;
    } else {
      const BoxGeom g = box_geom(false);
      if (!cache_map(&tmk, key_cache, c, hk, 16, g) ||
          !cache_map(&tmv, value_cache, c, kv_shared ? hk : hv, 16, g))
        return PA_ERR_CUDA;
    }
    if (TR >= 2 && mma_supported(hk, hv)) {
      err = launch_mma(tmk, tmv, P, n_items, stream);
    } else switch (TR) {
      case 1: err = launch_fma<1>(tmk, tmv, P, n_items, stream); break;
      case 2: err = launch_fma<2>(tmk, tmv, P, n_items, stream); break;
      case 3:
      case 4: err = launch_fma<4>(tmk, tmv, P, n_items, stream); break;
      default: err = launch_fma<8>(tmk, tmv, P, n_items, stream); break;
    }
  } else if (TR == PA_PF_TILE_ROWS || TR == PA_PF_PAIR_ROWS) {
    // rows meet many keys (more than one 64-row tile per kv head: 128-row
    // tiles, or 256-row tiles of two query tiles for prefill): 128-token key
    // tiles, boxes of the largest power of two (at most 128) dividing the
    // block size, both 64-dim halves in one box at 128
    const int rows = box_tokens(c.block_size, 128);
    const int halves = rows == 128 ? hk / 64 : 1;
    CUtensorMap tmk, tmv;
    if (!cache_map_3d(&tmk, key_cache, c, hk, rows, halves) ||
        !cache_map_3d(&tmv, value_cache, c, kv_shared ? hk : hv, rows, halves))
      return PA_ERR_CUDA;
    err = TR == PA_PF_PAIR_ROWS ? launch_pf_pair(tmk, tmv, P, n_items, stream)
                                : launch_pf(tmk, tmv, P, n_items, stream);
  } else if (tc_tile_rows(P.group, P.mask_q) == 16 && wide_supported(hk, hv, kv_shared)) {
    // 9-16 rows over a shared-KV cache: the 16-row warp-level MMA kernel,
    // 64-token tiles of every 64-dim block in one box (64-token boxes), else
    // one box per block piece and 64-dim block
    const int rows = box_tokens(c.block_size, 64);
    CUtensorMap tmk;
    if (!cache_map_3d(&tmk, key_cache, c, hk, rows, rows == 64 ? hk / 64 : 1)) return PA_ERR_CUDA;
    err = launch_wide(tmk, P, n_items, stream);
  } else {
    // 64-row tiles on the tcgen05 kernel: boxes of the largest power of two
    // (at most 64) dividing the block size
    if (!tc_supported(hk, hv)) return PA_ERR_UNSUPPORTED;
    const int rows = box_tokens(c.block_size, 64);
    const int halves = rows == 64 ? 2 : 1;
    CUtensorMap tmk, tmv, tmq;
    if (!cache_map_3d(&tmk, key_cache, c, hk, rows, halves) ||
        !cache_map_3d(&tmv, value_cache, c, kv_shared ? hk : hv, rows, halves))
      return PA_ERR_CUDA;
    // One query token per sequence (decode): a tile's rows are the G heads of
    // one kv head, consecutive in the query, so the producer fetches the tile
    // with TMA ahead of the K ring. Otherwise the softmax warps load it.
    P.q_tma = 0;
    tmq = tmk;
    if (max_q(c) == 1) {
      // one box for the whole tile when its rows are exactly the group's
      // (it lands as [block][G rows][128 B], the tile's layout), else one
      // box per 64-dim block
      const bool one_box = tc_tile_rows(P.group, P.mask_q) == P.group;
      if (!query_map(&tmq, query, c, one_box ? hk / 64 : 1)) return PA_ERR_CUDA;
      P.q_tma = one_box ? 2 : 1;
    }
    err = launch_tc(tmk, tmv, tmq, P, n_items, stream);
  }
  if (err != cudaSuccess) return PA_ERR_CUDA;
  if (n_combine > 0) {
    CombineParams C{};
    C.combine = combine;
    C.work = work;
    C.part_o = P.part_o;
    C.part_lse = P.part_lse;
    C.out = P.out;
    C.status = P.status;
    C.part_rows_cap = cap;
    C.num_heads = c.num_heads;
    C.group = P.group;
    C.hv = hv;
    C.counts = counts;
    if (launch_combine(C, n_combine, int(TR), stream) != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_forward(const pa_config* cfg, const void* query, const void* key_cache,
                                const void* value_cache, const int32_t* block_tables,
                                const int32_t* context_lens, const int32_t* q_seqlens,
                                const void* mask, const float* alibi_slopes, const int32_t* work,
                                int64_t n_items, const int32_t* combine, int64_t n_combine,
                                void* workspace, size_t workspace_bytes, void* out,
                                void* stream) {
  return forward_impl(cfg, query, key_cache, value_cache, block_tables, context_lens, q_seqlens,
                      mask, alibi_slopes, work, n_items, combine, n_combine, nullptr, workspace,
                      workspace_bytes, out, stream);
}

extern "C" pa_status pa_plan_bounds(const pa_config* cfg, int64_t* work_cap, int64_t* comb_cap,
                                    size_t* workspace_bytes) {
  using namespace pa;
  const pa_status st = validate_config(cfg);
  if (st != PA_OK) return st;
  const pa_config& c = *cfg;
  if (c.chunk_blocks < 0 || (c.chunk_blocks == 0 && c.num_sms <= 0)) return PA_ERR_INVALID_ARG;
  const int64_t TR = tile_rows(c);
  const int64_t rows = int64_t(c.num_heads / c.kv_heads) * max_q(c);
  const int64_t tiles = int64_t(c.batch) * c.kv_heads * cdiv(rows, TR);
  const int64_t items = c.chunk_blocks > 0 ? tiles * cdiv(c.max_blocks_per_seq, c.chunk_blocks)
                                           : 8 * int64_t(c.num_sms) + tiles;
  if (items > INT32_MAX || items * TR > INT32_MAX) return PA_ERR_INVALID_ARG;
  if (work_cap) *work_cap = items;
  if (comb_cap) *comb_cap = tiles;
  if (workspace_bytes) *workspace_bytes = workspace_layout(items * TR, c.head_size_v).total;
  return PA_OK;
}

extern "C" pa_status pa_plan_device(const pa_config* cfg, const int32_t* context_lens,
                                    const int32_t* q_seqlens, int32_t* work, int64_t work_cap,
                                    int32_t* combine, int64_t comb_cap, int32_t* counts,
                                    void* workspace, void* stream) {
  using namespace pa;
  const pa_status st = validate_config(cfg);
  if (st != PA_OK) return st;
  const pa_config& c = *cfg;
  if (!context_lens || !work || !counts || !workspace || (comb_cap > 0 && !combine))
    return PA_ERR_INVALID_ARG;
  if (c.chunk_blocks < 0 || (c.chunk_blocks == 0 && c.num_sms <= 0)) return PA_ERR_INVALID_ARG;
  if (work_cap < 1 || comb_cap < 0 || work_cap > INT32_MAX || comb_cap > INT32_MAX)
    return PA_ERR_INVALID_ARG;
  // the planner writes an item as two 16-byte stores, a combine entry as one
  if (!aligned(workspace, 256) || !aligned(work, 16) || (combine && !aligned(combine, 16)))
    return PA_ERR_INVALID_ARG;
  DevPlanParams D{};
  D.context_lens = context_lens;
  D.q_seqlens = q_seqlens;
  D.work = work;
  D.combine = combine;
  D.counts = counts;
  D.status = static_cast<uint32_t*>(workspace);
  D.work_cap = work_cap;
  D.comb_cap = comb_cap;
  D.batch = c.batch;
  D.num_heads = c.num_heads;
  D.kv_heads = c.kv_heads;
  D.group = c.num_heads / c.kv_heads;
  D.block_size = c.block_size;
  D.max_blocks_per_seq = c.max_blocks_per_seq;
  D.maxq = int(max_q(c));
  D.tr = int(tile_rows(c));
  D.chunk_blocks = c.chunk_blocks;
  D.num_sms = c.num_sms;
  D.hk = c.head_size_k;
  D.hv = c.head_size_v;
  return launch_plan(D, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_forward_device_plan(
    const pa_config* cfg, const void* query, const void* key_cache, const void* value_cache,
    const int32_t* block_tables, const int32_t* context_lens, const int32_t* q_seqlens,
    const void* mask, const float* alibi_slopes, const int32_t* work, int64_t work_cap,
    const int32_t* combine, int64_t comb_cap, const int32_t* counts, void* workspace,
    size_t workspace_bytes, void* out, void* stream) {
  if (!counts || work_cap < 1) return PA_ERR_INVALID_ARG;
  return forward_impl(cfg, query, key_cache, value_cache, block_tables, context_lens, q_seqlens,
                      mask, alibi_slopes, work, work_cap, combine, comb_cap, counts, workspace,
                      workspace_bytes, out, stream);
}

extern "C" pa_status pa_status_clear(void* workspace, void* stream) {
  if (!workspace) return PA_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

extern "C" pa_status pa_status_read(const void* workspace, void* stream_, uint32_t* bits) {
  if (!workspace) return PA_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return PA_ERR_CUDA;
  if (bits) *bits = v;
  if (v & PA_STATUS_BIT_TIMEOUT) return PA_ERR_TIMEOUT;
  if (v & PA_STATUS_BIT_BLOCK_INDEX) return PA_ERR_BLOCK_INDEX;
  if (v & PA_STATUS_BIT_WORKSPACE) return PA_ERR_BUFFER_TOO_SMALL;
  if (v & PA_STATUS_BIT_PLAN) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

extern "C" pa_status pa_testing_set_wait_limit(long long cycles) {
  if (cycles < 0) return PA_ERR_INVALID_ARG;
  pa::g_wait_limit.store(cycles, std::memory_order_relaxed);
  return PA_OK;
}

extern "C" const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported mode";
    case PA_ERR_BUFFER_TOO_SMALL: return "buffer too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_BLOCK_INDEX: return "block table entry out of range";
    case PA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}
