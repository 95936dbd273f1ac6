// Pieces shared by the warp-pipelined decode kernels (CUDA-core and mma.sync):
// the work item, the per-warp TMA pipeline over 16-token sub-tiles, the
// shared-memory layout, and the cross-warp softmax merge with the final store.
//
// A work item (pa.h) is one (sequence, kv head, row tile, KV-block range).
// Its tokens are cut into 16-token sub-tiles; warp w of the CTA owns
// sub-tiles w, w + NW, w + 2 NW, ... and streams them through its own ring of
// NBUF shared-memory buffers with 2-D TMA copies (one box per 64 or 16 head
// dims, 128- or 32-byte swizzle), each buffer completing on its own mbarrier.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kSubTokens = 16;  // tokens per sub-tile = TMA box height

struct Item {
  int b, kvh, r0, r1, kb0, kb1, q_start, slot;
  int nrows, L, qlen, tok0, tok1, nsub;

  __device__ __forceinline__ void load(const FwdParams& P, int idx) {
    const int32_t* it = P.work + int64_t(idx) * PA_WORK_INTS;
    b = it[0];
    kvh = it[1];
    r0 = it[2];
    r1 = it[3];
    kb0 = it[4];
    kb1 = it[5];
    q_start = it[6];
    slot = it[7];
    nrows = r1 - r0;
    L = P.context_lens[b];
    qlen = P.q_seqlens ? P.q_seqlens[b] : 1;
    tok0 = kb0 * P.block_size;
    tok1 = min(kb1 * P.block_size, L);
    nsub = tok1 > tok0 ? (tok1 - tok0 + kSubTokens - 1) / kSubTokens : 0;
  }
};

// Floats per warp in the merge area: m[rt], l[rt] padded to 4, then O[rt][hv].
__host__ __device__ inline uint32_t merge_stride(int rt, int hv) {
  return uint32_t((2 * rt + 3) / 4 * 4 + rt * hv);
}
__host__ __device__ inline int merge_opart(int rt) { return (2 * rt + 3) / 4 * 4; }

struct PipeLayout {
  uint32_t front;       // kernel-specific bytes after the barriers
  uint32_t buf_off;     // first buffer
  uint32_t buf_stride;  // bytes per buffer (K then V, 1024-aligned)
  uint32_t v_in_buf;    // offset of V inside a buffer
  uint32_t bytes;       // dynamic shared memory to request
};

// [128 B barriers][front][NW * NBUF buffers]; the merge area aliases the
// buffers once every warp has finished streaming.
__host__ __device__ inline PipeLayout pipe_layout(int nw, int nbuf, int hk, int hv, uint32_t front,
                                                  int merge_rt) {
  auto up = [](uint32_t x, uint32_t a) { return (x + a - 1) / a * a; };
  PipeLayout L;
  L.front = front;
  L.buf_off = up(128 + front, 1024);
  L.v_in_buf = up(uint32_t(kSubTokens) * hk * 2, 1024);
  L.buf_stride = up(L.v_in_buf + uint32_t(kSubTokens) * hv * 2, 1024);
  const uint32_t bufs_end = L.buf_off + uint32_t(nw) * nbuf * L.buf_stride;
  const uint32_t merge_end = L.buf_off + uint32_t(nw) * merge_stride(merge_rt, hv) * 4;
  L.bytes = (bufs_end > merge_end ? bufs_end : merge_end) + 1024;  // + base alignment slack
  return L;
}

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// One warp's TMA ring. All member functions are warp-collective except where
// noted; lane 0 issues the copies.
template <int KBW, int VBW, int NBUF>
struct WarpPipe {
  static constexpr uint32_t kBoxBytes = uint32_t(kSubTokens) * KBW * 2;
  static constexpr uint32_t vBoxBytes = uint32_t(kSubTokens) * VBW * 2;

  uint64_t* bars;
  uint8_t* bufs;
  uint32_t stride, v_off, tile_bytes;
  const int32_t* bt_row;
  int bt_base, bt_reg;
  int kb0, kb1, warp, nw, lane, bs, hk, hv, kvh, num_blocks, nkbox, nvbox;
  bool shared;  // V is read from the K boxes (shared-KV cache): no V copies
  uint32_t* status;
  long long wait_limit;
  uint64_t pol;
  const CUtensorMap* tmk;
  const CUtensorMap* tmv;

  __device__ __forceinline__ void init(uint8_t* smem, const PipeLayout& lay, const FwdParams& P,
                                       const Item& it, const CUtensorMap* k_map,
                                       const CUtensorMap* v_map) {
    lane = threadIdx.x & 31;
    warp = threadIdx.x >> 5;
    nw = blockDim.x >> 5;
    bars = reinterpret_cast<uint64_t*>(smem) + warp * NBUF;
    bufs = smem + lay.buf_off + uint32_t(warp) * NBUF * lay.buf_stride;
    stride = lay.buf_stride;
    v_off = lay.v_in_buf;
    hk = P.hk;
    hv = P.hv;
    shared = P.kv_shared != 0;
    tile_bytes = uint32_t(kSubTokens) * (hk + (shared ? 0 : hv)) * 2;
    nkbox = hk / KBW;
    nvbox = hv / VBW;
    bs = P.block_size;
    kvh = it.kvh;
    kb0 = it.kb0;
    kb1 = it.kb1;
    num_blocks = P.num_blocks;
    status = P.status;
    wait_limit = P.wait_limit;
    tmk = k_map;
    tmv = v_map;
    pol = policy_evict_first();
    if (lane == 0) {
      for (int k = 0; k < NBUF; ++k) mbar_init(&bars[k], 1);
      fence_barrier_init();
    }
    __syncwarp();
    // Block-table window: lane k holds the entry of block kb0 + bt_base + k.
    bt_row = P.block_tables + int64_t(it.b) * P.max_blocks_per_seq;
    bt_base = 0;
    bt_reg = (kb0 + lane < kb1) ? bt_row[kb0 + lane] : 0;
  }

  // Sub-tile index (within the item) of this warp's n-th sub-tile.
  __device__ __forceinline__ int sub(int n) const { return warp + n * nw; }
  __device__ __forceinline__ uint8_t* kbuf(int n) const { return bufs + (n % NBUF) * stride; }
  // With a shared-KV cache the V sub-tile is the first hv / VBW boxes of the
  // K sub-tile (K and V boxes have the same width, so the same layout).
  __device__ __forceinline__ uint8_t* vbuf(int n) const { return shared ? kbuf(n) : kbuf(n) + v_off; }

  // Start the copies of this warp's n-th sub-tile into buffer n % NBUF.
  __device__ __forceinline__ void issue(int n) {
    const int u = sub(n);
    const int rel = (u * kSubTokens) / bs;
    const int off = (u * kSubTokens) % bs;
    if (rel >= bt_base + 32) {
      bt_base = rel & ~31;
      bt_reg = (kb0 + bt_base + lane < kb1) ? bt_row[kb0 + bt_base + lane] : 0;
    }
    const int phys = __shfl_sync(0xffffffffu, bt_reg, rel - bt_base);
    if (lane == 0) {
      uint64_t* bar = &bars[n % NBUF];
      if (phys < 0 || phys >= num_blocks) {
        // Never dereference a bad entry: flag it and complete the phase
        // without a copy (the buffer keeps stale data; the status word says
        // the result is invalid).
        set_status(status, PA_STATUS_BIT_BLOCK_INDEX);
        mbar_arrive(bar);
        return;
      }
      const int row = phys * bs + off;
      uint8_t* dst = kbuf(n);
      mbar_arrive_expect_tx(bar, tile_bytes);
      if constexpr (KBW == 64 && VBW == 64) {
        // 64-dim blocks: one 3-D box per sub-tile and cache, landing as the
        // same [block][16 tokens][128 B] sequence the 2-D boxes would (fewer,
        // larger copies: each costs the issuing lane time on a busy SM)
        tma_load_3d(dst, tmk, bar, 0, row, kvh * nkbox, pol);
        if (!shared) tma_load_3d(dst + v_off, tmv, bar, 0, row, kvh * nvbox, pol);
      } else {
        for (int j = 0; j < nkbox; ++j)
          tma_load_2d(dst + j * kBoxBytes, tmk, bar, kvh * hk + j * KBW, row, pol);
        if (!shared)
          for (int j = 0; j < nvbox; ++j)
            tma_load_2d(dst + v_off + j * vBoxBytes, tmv, bar, kvh * hv + j * VBW, row, pol);
      }
    }
  }

  // Bounded wait for the n-th sub-tile, warp-collective: every lane waits
  // (each lane then reads the buffer), and the verdict is the warp's, so that
  // a lane whose wait ran out and one whose copy landed meanwhile cannot part.
  __device__ __forceinline__ bool wait(int n) {
    return __all_sync(0xffffffffu, mbar_wait_own(&bars[n % NBUF], (n / NBUF) & 1, wait_limit));
  }

  // Called by the warp once it is done reading buffer n % NBUF.
  __device__ __forceinline__ void release_and_refill(int n, int nmine) {
    __syncwarp();
    fence_proxy_async();
    if (n + NBUF < nmine) issue(n + NBUF);
  }

  // After a timed-out wait at sub-tile `failed`: let the copies still in
  // flight (sub-tiles failed .. failed + NBUF - 1, the ones issued and not yet
  // consumed) land before the CTA's shared memory is released. These waits
  // take the default limit whatever wait_limit is: the copies were issued and
  // land within microseconds.
  __device__ __forceinline__ void drain(int failed, int nmine) {
    if (lane == 0) set_status(status, PA_STATUS_BIT_TIMEOUT);
    for (int m = failed; m < failed + NBUF && m < nmine; ++m)
      mbar_wait(&bars[m % NBUF], (m / NBUF) & 1);
  }
};

// Merge the per-warp softmax states (m, l in base 2; O unnormalised) stored at
// `base` with stride merge_stride(RT, hv), and write the tile's rows: fp16
// output when the item is unsplit, else fp16 partial rows and their fp32
// natural-log LSE. Called by the whole CTA after a __syncthreads.
template <int RT>
__device__ __forceinline__ void merge_store(const FwdParams& P, const Item& it, const float* base,
                                            int nw) {
  const int hv = P.hv, G = P.group;
  const int mstride = int(merge_stride(RT, hv)), opart = merge_opart(RT);
  const bool partial = it.slot >= 0;
  if (partial && int64_t(it.slot) + it.nrows > P.part_rows_cap) {
    if (threadIdx.x == 0) set_status(P.status, PA_STATUS_BIT_WORKSPACE);
    return;
  }
  for (int idx = threadIdx.x; idx < it.nrows * hv; idx += blockDim.x) {
    const int rr = idx / hv, d = idx % hv;
    float M = -INFINITY;
    for (int w = 0; w < nw; ++w) M = fmaxf(M, base[w * mstride + rr]);
    float lsum = 0.f, osum = 0.f;
    for (int w = 0; w < nw; ++w) {
      const float* ww = base + w * mstride;
      const float f = ex2(ww[rr] - M);
      lsum += ww[RT + rr] * f;
      osum += ww[opart + rr * hv + d] * f;
    }
    const float val = osum / lsum;
    if (!partial) {
      const int r = it.r0 + rr, i = r / G, h = it.kvh * G + r % G;
      P.out[(int64_t(it.q_start + i) * P.num_heads + h) * hv + d] = __float2half_rn(val);
    } else {
      P.part_o[(int64_t(it.slot) + rr) * hv + d] = __float2half_rn(val);
      if (d == 0) P.part_lse[it.slot + rr] = (M + log2f(lsum)) * kLn2;
    }
  }
}

}  // namespace pa
