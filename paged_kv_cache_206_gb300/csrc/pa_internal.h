// Host-side helpers shared by the planner and the launch code of libpa.so.
#pragma once

#include <cstdint>

#include "pa.h"

namespace pa {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Checks of a pa_config against the operator's constraints (block_size % 16,
// batch limit, GQA divisibility, head-size range, block_size <= 128 for head
// sizes above 256 and for parallel decoding) and this library's own rules
// (head sizes multiple of 16, supported mask types).
pa_status validate_config(const pa_config* cfg);

inline int64_t max_q(const pa_config& c) { return c.max_seqlen_q > 0 ? c.max_seqlen_q : 1; }

// Tokens per TMA box of a kernel with `tile`-token key tiles (a power of two):
// the largest power of two dividing both the block size and the tile, so that
// no box crosses from one block into the next physical one. The kernels derive
// the same figure from the block size.
inline int box_tokens(int block_size, int tile) {
  const int p2 = block_size & -block_size;
  return p2 < tile ? p2 : tile;
}

// The host-side checks of pa_forward (configuration, pointers, alignment,
// workspace size), done before anything is enqueued; the workspace pointer
// itself is checked (non-null, 256-byte aligned) only with check_workspace.
pa_status check_forward(const pa_config* cfg, const void* query, const void* key_cache,
                        const void* value_cache, const int32_t* block_tables,
                        const int32_t* context_lens, const void* mask, const float* alibi_slopes,
                        const int32_t* work, int64_t n_items, const int32_t* combine,
                        int64_t n_combine, const void* workspace, size_t workspace_bytes,
                        const void* out, bool check_workspace);

// Tile height of a launch: every row of a (b, kv head) pair in one CTA when
// the group is small enough for the CUDA-core kernel; for 64/128-dim heads
// with more than 64 rows, 128-row tiles, or 256 (two 128-row query tiles
// sharing K and V) past 128 rows; else 64-row tiles.
inline int64_t tile_rows(const pa_config& c) {
  const int64_t g = c.num_heads / c.kv_heads;
  const int64_t r = g * max_q(c);
  if (r <= PA_FMA_MAX_ROWS) return r;
  const bool pf_heads = c.head_size_k == c.head_size_v && (c.head_size_k == 64 || c.head_size_k == 128);
  if (r > PA_TC_TILE_ROWS && pf_heads) return r > PA_PF_TILE_ROWS ? PA_PF_PAIR_ROWS : PA_PF_TILE_ROWS;
  return PA_TC_TILE_ROWS;
}

#ifdef __CUDACC__
#define PA_HOST_DEVICE __host__ __device__
#else
#define PA_HOST_DEVICE
#endif

// Last chunk the wave fit of the automatic chunk rule tries after the
// balance chunk c0: at most twice c0, at most 31 past it, and none past the
// longest sequence's block count (from there on every chunk gives the same
// items, so a longer one only costs).
PA_HOST_DEVICE inline int64_t wave_fit_hi(int64_t c0, int64_t max_nb) {
  int64_t hi = 2 * c0 < c0 + 31 ? 2 * c0 : c0 + 31;
  const int64_t cap = max_nb > c0 ? max_nb : c0;
  return hi < cap ? hi : cap;
}

struct WorkspaceLayout {
  size_t partial_o;    // byte offset of the fp16 [P, hv] partial outputs
  size_t partial_lse;  // byte offset of the fp32 [P] log-sum-exps
  size_t total;        // bytes
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// [status][partial O][partial LSE], each part on a 256-byte boundary.
inline WorkspaceLayout workspace_layout(int64_t partial_rows, int hv) {
  WorkspaceLayout w;
  w.partial_o = PA_STATUS_BYTES;
  w.partial_lse = align256(w.partial_o + size_t(partial_rows) * size_t(hv) * 2);
  w.total = align256(w.partial_lse + size_t(partial_rows) * 4);
  return w;
}

// Partial rows that a workspace of `bytes` can hold for value head size hv.
inline int64_t workspace_rows(size_t bytes, int hv) {
  if (bytes < PA_STATUS_BYTES) return -1;
  // largest P with workspace_layout(P, hv).total <= bytes
  int64_t lo = 0, hi = int64_t((bytes - PA_STATUS_BYTES) / (size_t(hv) * 2 + 4)) + 1;
  while (lo + 1 < hi) {
    const int64_t mid = (lo + hi) / 2;
    if (workspace_layout(mid, hv).total <= bytes) lo = mid; else hi = mid;
  }
  return lo;
}

}  // namespace pa
