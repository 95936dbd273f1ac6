// Host planner of libpa.so: constraint checks and the split-KV work list.
//
// The work list restates the task list of SparseAttnSharedkvMetadata
// ("功能说明" and its `metadata` output): per CTA the batch, head group, query
// tile and KV-block range it computes, plus the reduction tasks that merge
// split results. The exact rule (tile height, chunk size, order, slots) is
// written out in pa.h.
#include <cmath>
#include <algorithm>
#include <cstring>
#include <initializer_list>

#include "pa_internal.h"

namespace pa {

pa_status validate_config(const pa_config* cfg) {
  if (!cfg) return PA_ERR_INVALID_ARG;
  const pa_config& c = *cfg;
  // PagedAttentionOperation "Constraints": 0 < batch <= 2048.
  if (c.batch <= 0 || c.batch > PA_MAX_BATCH) return PA_ERR_INVALID_ARG;
  // GQA: headNum % kvHeadNum == 0 (equal counts are plain MHA).
  if (c.num_heads <= 0 || c.kv_heads <= 0 || c.num_heads % c.kv_heads) return PA_ERR_INVALID_ARG;
  // Head sizes in (0, 576]; ours: multiples of 16 (16-byte vectors, TMA rows).
  for (int hs : {c.head_size_k, c.head_size_v})
    if (hs <= 0 || hs > PA_MAX_HEAD_SIZE || hs % 16) return PA_ERR_INVALID_ARG;
  // block_size % 16 == 0.
  if (c.block_size <= 0 || c.block_size % 16) return PA_ERR_INVALID_ARG;
  // A head size above 256 needs block_size <= 128; so does parallel decoding.
  if ((c.head_size_k > 256 || c.head_size_v > 256) && c.block_size > 128) return PA_ERR_INVALID_ARG;
  if (max_q(c) > 1 && c.block_size > 128) return PA_ERR_INVALID_ARG;
  if (c.num_blocks <= 0 || c.max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
  // TMA row coordinates are int32.
  if (int64_t(c.num_blocks) * c.block_size > INT32_MAX) return PA_ERR_INVALID_ARG;
  if (c.max_seqlen_q < 0) return PA_ERR_INVALID_ARG;
  switch (c.mask_type) {
    case PA_MASK_NONE:
    case PA_MASK_ALIBI:
    case PA_MASK_NORM:
      break;
    case PA_MASK_NORM_COMPRESS:
      if (max_q(c) > PA_COMPRESS_MASK_SIZE) return PA_ERR_INVALID_ARG;
      break;
    case PA_MASK_SPEC:
      return PA_ERR_UNSUPPORTED;
    default:
      return PA_ERR_INVALID_ARG;
  }
  if (c.chunk_blocks < 0) return PA_ERR_INVALID_ARG;
  if (c.chunk_blocks == 0 && c.num_sms <= 0) return PA_ERR_INVALID_ARG;
  if (std::isnan(c.scale) || std::isinf(c.scale)) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

}  // namespace pa

using pa::cdiv;

extern "C" pa_status pa_plan(const pa_config* cfg, const int32_t* context_lens,
                             const int32_t* q_seqlens, int32_t* work, int64_t work_cap,
                             int64_t* n_items, int32_t* combine, int64_t comb_cap,
                             int64_t* n_combine, size_t* workspace_bytes) {
  pa_status st = pa::validate_config(cfg);
  if (st != PA_OK) return st;
  if (!context_lens) return PA_ERR_INVALID_ARG;
  const pa_config& c = *cfg;
  const int64_t Hk = c.kv_heads, G = c.num_heads / c.kv_heads, bs = c.block_size;
  const int64_t TR = pa::tile_rows(c), maxq = pa::max_q(c);

  // Per-sequence checks, and the work measure of the automatic chunk rule.
  int64_t W = 0, total_q = 0, maxNB = 0;
  for (int b = 0; b < c.batch; ++b) {
    const int64_t L = context_lens[b];
    const int64_t q = q_seqlens ? q_seqlens[b] : 1;
    if (q < 1 || q > maxq) return PA_ERR_INVALID_ARG;
    if (L < q) return PA_ERR_INVALID_ARG;  // kvSeqLen >= qSeqLen, and so L >= 1
    const int64_t NB = cdiv(L, bs);
    // max_num_blocks_per_seq >= ceil(max(contextLens) / block_size)
    if (NB > c.max_blocks_per_seq) return PA_ERR_INVALID_ARG;
    W += NB * Hk * cdiv(G * q, TR);
    total_q += q;
    maxNB = std::max(maxNB, NB);
  }
  if (total_q * c.num_heads > INT32_MAX) return PA_ERR_INVALID_ARG;

  int64_t chunk;
  if (c.chunk_blocks > 0) {
    chunk = c.chunk_blocks;
  } else {
    // items per SM aimed at: 8 for the warp kernels (several CTAs per SM), 2
    // for the tcgen05 kernel (one CTA per SM, a longer fixed cost per item)
    const int64_t per_sm = TR <= PA_FMA_MAX_ROWS ? 8 : 2;
    const int64_t bal = cdiv(W, per_sm * int64_t(c.num_sms));
    const int64_t RT = std::min(TR, G * maxq);  // rows a full tile really holds
    const int64_t lo = cdiv(64 * RT * c.head_size_v, bs * (c.head_size_k + c.head_size_v));
    chunk = std::max<int64_t>(1, std::max(bal, lo));
    if (TR > PA_FMA_MAX_ROWS) {
      // One CTA per SM: items run in waves of num_sms. Of the chunks
      // chunk .. wave_fit_hi(chunk, maxNB), take the one with the least
      // waves x chunk (the first on a tie).
      const int64_t hi = pa::wave_fit_hi(chunk, maxNB);
      int64_t best = chunk, best_cost = -1;
      for (int64_t cc = chunk; cc <= hi; ++cc) {
        int64_t n = 0;
        for (int b = 0; b < c.batch; ++b) {
          const int64_t q = q_seqlens ? q_seqlens[b] : 1;
          n += Hk * cdiv(G * q, TR) * cdiv(cdiv(context_lens[b], bs), cc);
        }
        const int64_t cost = cdiv(n, int64_t(c.num_sms)) * cc;
        if (best_cost < 0 || cost < best_cost) {
          best_cost = cost;
          best = cc;
        }
      }
      chunk = best;
    }
  }

  // Counts.
  int64_t items = 0, combines = 0, prows = 0;
  for (int b = 0; b < c.batch; ++b) {
    const int64_t q = q_seqlens ? q_seqlens[b] : 1;
    const int64_t R = G * q, QT = cdiv(R, TR);
    const int64_t S = cdiv(cdiv(context_lens[b], bs), chunk);
    items += Hk * QT * S;
    if (S > 1) {
      combines += Hk * QT;
      prows += Hk * S * R;  // the tiles of one (b, kvh) hold R rows in total
    }
  }
  if (items > INT32_MAX || prows > INT32_MAX) return PA_ERR_INVALID_ARG;
  if (n_items) *n_items = items;
  if (n_combine) *n_combine = combines;
  if (workspace_bytes) *workspace_bytes = pa::workspace_layout(prows, c.head_size_v).total;
  if ((work && work_cap < items) || (combine && comb_cap < combines)) return PA_ERR_BUFFER_TOO_SMALL;
  if (!work && !combine) return PA_OK;

  // Lists, in (b, kvh, qt, split) order.
  int64_t it = 0, ce = 0, slot = 0, q_start = 0;
  for (int b = 0; b < c.batch; ++b) {
    const int64_t q = q_seqlens ? q_seqlens[b] : 1;
    const int64_t R = G * q, QT = cdiv(R, TR);
    const int64_t NB = cdiv(context_lens[b], bs);
    const int64_t S = cdiv(NB, chunk);
    for (int64_t kvh = 0; kvh < Hk; ++kvh) {
      for (int64_t qt = 0; qt < QT; ++qt) {
        const int64_t r0 = qt * TR, r1 = std::min(R, r0 + TR);
        if (S > 1) {
          if (combine) {
            int32_t* e = combine + ce * PA_COMBINE_INTS;
            e[0] = b;
            e[1] = int32_t(kvh);
            e[2] = int32_t(it);
            e[3] = int32_t(S);
          }
          ++ce;
        }
        for (int64_t s = 0; s < S; ++s, ++it) {
          if (work) {
            int32_t* w = work + it * PA_WORK_INTS;
            w[0] = b;
            w[1] = int32_t(kvh);
            w[2] = int32_t(r0);
            w[3] = int32_t(r1);
            w[4] = int32_t(s * chunk);
            w[5] = int32_t(std::min(NB, (s + 1) * chunk));
            w[6] = int32_t(q_start);
            w[7] = S > 1 ? int32_t(slot) : -1;
          }
          if (S > 1) slot += r1 - r0;
        }
      }
    }
    q_start += q;
  }
  return PA_OK;
}
