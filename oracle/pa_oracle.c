/*
 * pa_oracle.c -- CPU reference for paged attention, in double precision.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this code; the library's product path never does.
 * It shares no code, header or table with the CUDA path.
 *
 * oracle_attention follows the PagedAttentionOperation pages literally:
 *   1. resolve the block table of a sequence into contiguous K and V
 *      ("Constraints": blockTables rows index physical blocks of
 *      block_size tokens; contextLens is the whole KV length);
 *   2. score every visible key, add the mask or bias, and take a textbook
 *      softmax (subtract the max, exponentiate, sum, divide);
 *   3. weight V by the softmax.
 * Readings where the pages are silent:
 *   - GQA head h reads kv head h / (H / Hk);
 *   - s = scale * <q, k> + bias; the bias is not scaled;
 *   - query token i of a sequence sits at position p = L - q + i
 *     (prefix = max(0, kvSeqLen - qSeqLen), MASK_TYPE_NORM_COMPRESS bullets);
 *   - the compressed 2048 x 2048 mask is applied with the shift
 *     sigma = max(0, L - 2048): bias = mask[p - sigma][j - sigma] for
 *     j >= sigma, else 0 (it "adapts automatically" to longer sequences);
 *   - ALiBi bias = slope_h * (j - p);
 *   - MASK_TYPE_NORM (the model's own mask, "How to select a mask") is an
 *     explicit additive tensor per sequence: bias = mask[b][i][j] for query
 *     token i and key j, the tensor being [batch][mask_q][mask_kv] with
 *     mask_q = max_seqlen_q and mask_kv = max_blocks_per_seq * block_size.
 * The oracle reads the whole mask row it needs, lower triangle included; for a
 * mask as the pages define it that part is zero. For mask tensors that break
 * that definition the oracle and the kernels may differ: parity unpinned there.
 *
 * oracle_plan restates the work-list rule (task list of
 * SparseAttnSharedkvMetadata, "功能说明" / `metadata`) as the header of the
 * library words it, without sharing its code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, from the format's definition. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(frac + 1024), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
  }
  return sign ? -v : v;
}

enum { MASK_NONE = 0, MASK_NORM = 1, MASK_ALIBI = 2, MASK_NORM_COMPRESS = 5 };
#define MASK_DIM 2048

typedef struct {
  int batch, num_heads, kv_heads, hk, hv, block_size, num_blocks, max_blocks_per_seq;
  int mask_type;
  double scale;
  int64_t mask_q, mask_kv; /* MASK_NORM tensor dims after the batch */
} oracle_shape;

/* One (sequence, kv head) unit: gather, then every head of the group and
 * every query token of the sequence. */
static void unit(const oracle_shape* S, int b, int kvh, const uint16_t* query,
                 const uint16_t* key_cache, const uint16_t* value_cache,
                 const int32_t* block_tables, const int32_t* context_lens,
                 const int64_t* q_start, const int32_t* q_seqlens, const uint16_t* mask,
                 const float* alibi_slopes, double* out) {
  const int L = context_lens[b];
  const int q = q_seqlens ? q_seqlens[b] : 1;
  const int G = S->num_heads / S->kv_heads;
  const int hk = S->hk, hv = S->hv, bs = S->block_size, Hk = S->kv_heads, H = S->num_heads;
  double* K = (double*)malloc(sizeof(double) * (size_t)L * hk);
  double* V = (double*)malloc(sizeof(double) * (size_t)L * hv);
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  /* 1. resolve the block table: logical token j lives in physical block
   *    block_tables[b][j / bs] at slot j % bs. */
  for (int j = 0; j < L; ++j) {
    int64_t phys = block_tables[(int64_t)b * S->max_blocks_per_seq + j / bs];
    int64_t slot = j % bs;
    const uint16_t* kr = key_cache + ((phys * bs + slot) * Hk + kvh) * hk;
    const uint16_t* vr = value_cache + ((phys * bs + slot) * Hk + kvh) * hv;
    for (int d = 0; d < hk; ++d) K[(size_t)j * hk + d] = oracle_half_to_double(kr[d]);
    for (int d = 0; d < hv; ++d) V[(size_t)j * hv + d] = oracle_half_to_double(vr[d]);
  }
  const int sigma = L > MASK_DIM ? L - MASK_DIM : 0;
  for (int g = 0; g < G; ++g) {
    const int h = kvh * G + g;
    for (int i = 0; i < q; ++i) {
      const int p = L - q + i;
      const int64_t row = (q_start[b] + i) * H + h;
      const uint16_t* qr = query + row * hk;
      double qd[1024];
      for (int d = 0; d < hk; ++d) qd[d] = oracle_half_to_double(qr[d]);
      /* 2. scores with mask or bias */
      for (int j = 0; j < L; ++j) {
        double dot = 0.0;
        for (int d = 0; d < hk; ++d) dot += qd[d] * K[(size_t)j * hk + d];
        double bias = 0.0;
        if (S->mask_type == MASK_ALIBI) {
          bias = (double)alibi_slopes[h] * (double)(j - p);
        } else if (S->mask_type == MASK_NORM_COMPRESS) {
          if (j >= sigma)
            bias = oracle_half_to_double(mask[(int64_t)(p - sigma) * MASK_DIM + (j - sigma)]);
        } else if (S->mask_type == MASK_NORM) {
          bias = oracle_half_to_double(mask[((int64_t)b * S->mask_q + i) * S->mask_kv + j]);
        }
        s[j] = S->scale * dot + bias;
      }
      /* textbook softmax */
      double m = -INFINITY;
      for (int j = 0; j < L; ++j) m = s[j] > m ? s[j] : m;
      double sum = 0.0;
      for (int j = 0; j < L; ++j) {
        s[j] = exp(s[j] - m);
        sum += s[j];
      }
      /* 3. weight the values */
      double* o = out + row * hv;
      for (int d = 0; d < hv; ++d) o[d] = 0.0;
      for (int j = 0; j < L; ++j) {
        const double w = s[j] / sum;
        for (int d = 0; d < hv; ++d) o[d] += w * V[(size_t)j * hv + d];
      }
    }
  }
  free(K);
  free(V);
  free(s);
}

/*
 * Attention for the sequences listed in `subset` (all sequences when subset is
 * NULL). `out` is double [sum q_b, H, hv]; rows of sequences outside the subset
 * are left untouched. `threads` > 0 sets the OpenMP thread count. Returns the
 * number of threads used.
 */
int oracle_attention(int batch, int num_heads, int kv_heads, int hk, int hv, int block_size,
                     int num_blocks, int max_blocks_per_seq, int mask_type, double scale,
                     const uint16_t* query, const uint16_t* key_cache,
                     const uint16_t* value_cache, const int32_t* block_tables,
                     const int32_t* context_lens, const int32_t* q_seqlens,
                     const uint16_t* mask, int64_t mask_q, int64_t mask_kv,
                     const float* alibi_slopes, const int32_t* subset, int n_subset,
                     double* out, int threads) {
  oracle_shape S = {batch, num_heads, kv_heads, hk, hv, block_size, num_blocks,
                    max_blocks_per_seq, mask_type, scale, mask_q, mask_kv};
  if (hk > 1024) return -1;
  int64_t* q_start = (int64_t*)malloc(sizeof(int64_t) * (size_t)(batch + 1));
  q_start[0] = 0;
  for (int b = 0; b < batch; ++b) q_start[b + 1] = q_start[b] + (q_seqlens ? q_seqlens[b] : 1);
  const int nb = subset ? n_subset : batch;
  const int64_t units = (int64_t)nb * kv_heads;
  int used = 1;
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel
  {
#pragma omp single
    used = omp_get_num_threads();
#pragma omp for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
      const int bi = (int)(u / kv_heads);
      const int b = subset ? subset[bi] : bi;
      unit(&S, b, (int)(u % kv_heads), query, key_cache, value_cache, block_tables,
           context_lens, q_start, q_seqlens, mask, alibi_slopes, out);
    }
  }
#else
  (void)threads;
  for (int64_t u = 0; u < units; ++u) {
    const int bi = (int)(u / kv_heads);
    const int b = subset ? subset[bi] : bi;
    unit(&S, b, (int)(u % kv_heads), query, key_cache, value_cache, block_tables, context_lens,
         q_start, q_seqlens, mask, alibi_slopes, out);
  }
#endif
  free(q_start);
  if (units < used) used = (int)units;
  return used;
}

/* ceil(a / b) for positive integers */
static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

/*
 * The work-list rule, restated from its written definition:
 *   tile height    TR = G * maxq if that is at most 8; else, when hk = hv in
 *                  {64, 128}, 256 if G * maxq > 128 and 128 if G * maxq > 64;
 *                  else 64
 *   tiles          QT_b = ceil(G * q_b / TR)
 *   blocks         NB_b = ceil(L_b / bs)
 *   chunk          c = chunk_blocks if positive, else
 *                  max(1, ceil(sum_b NB_b*Hk*QT_b / (k*num_sms)),
 *                         ceil(64*RT*hv / (bs*(hk+hv))))
 *                  with RT = min(TR, G * maxq), the rows a full tile holds,
 *                  and k = 8 when TR <= 8, else 2; then, when TR > 8 (one CTA
 *                  per SM), the wave fit: of c0 = that value and the chunks
 *                  up to min(2*c0, c0 + 31, max(c0, max_b NB_b)), the one with
 *                  the least ceil(items(c) / num_sms) * c, the first on a tie
 *   splits         S_b = ceil(NB_b / c); split s = blocks [s*c, min(NB_b, (s+1)*c))
 *   items          (b, kvh, qt, s) lexicographic; 8 ints
 *                  {b, kvh, row_begin, row_end, kb_begin, kb_end, q_start, slot}
 *   slots          running count of partial rows over items with S_b > 1
 *   combine        one {b, kvh, first_item, S_b} per (b, kvh, qt) with S_b > 1
 * Counts are always written; lists only when the pointers are non-NULL and
 * the capacities suffice. Returns 0, or 1 when a capacity is too small.
 */
int oracle_plan(int batch, int num_heads, int kv_heads, int hk, int hv, int block_size,
                int max_seqlen_q, int chunk_blocks, int num_sms, const int32_t* context_lens,
                const int32_t* q_seqlens, int32_t* work, int64_t work_cap, int64_t* n_items,
                int32_t* comb, int64_t comb_cap, int64_t* n_comb, int64_t* n_partial_rows) {
  const int64_t G = num_heads / kv_heads;
  const int64_t maxq = max_seqlen_q > 0 ? max_seqlen_q : 1;
  int64_t TR = 64;
  if (G * maxq <= 8) TR = G * maxq;
  else if (G * maxq > 64 && hk == hv && (hk == 64 || hk == 128)) TR = G * maxq > 128 ? 256 : 128;
  int64_t c;
  if (chunk_blocks > 0) {
    c = chunk_blocks;
  } else {
    int64_t W = 0;
    for (int b = 0; b < batch; ++b) {
      const int64_t q = q_seqlens ? q_seqlens[b] : 1;
      W += cdiv(context_lens[b], block_size) * kv_heads * cdiv(G * q, TR);
    }
    const int64_t per_sm = TR <= 8 ? 8 : 2;
    const int64_t c_bal = cdiv(W, per_sm * (int64_t)num_sms);
    const int64_t RT = TR < G * maxq ? TR : G * maxq;
    const int64_t c_min = cdiv(64 * RT * hv, (int64_t)block_size * (hk + hv));
    c = 1;
    if (c_bal > c) c = c_bal;
    if (c_min > c) c = c_min;
    if (TR > 8) {
      int64_t max_nb = 0;
      for (int b = 0; b < batch; ++b) {
        const int64_t nb = cdiv(context_lens[b], block_size);
        if (nb > max_nb) max_nb = nb;
      }
      int64_t last = 2 * c;
      if (c + 31 < last) last = c + 31;
      if ((max_nb > c ? max_nb : c) < last) last = max_nb > c ? max_nb : c;
      int64_t best = c, best_cost = -1;
      for (int64_t cand = c; cand <= last; ++cand) {
        int64_t n = 0;
        for (int b = 0; b < batch; ++b) {
          const int64_t q = q_seqlens ? q_seqlens[b] : 1;
          n += kv_heads * cdiv(G * q, TR) * cdiv(cdiv(context_lens[b], block_size), cand);
        }
        const int64_t cost = cdiv(n, (int64_t)num_sms) * cand;
        if (best_cost < 0 || cost < best_cost) {
          best_cost = cost;
          best = cand;
        }
      }
      c = best;
    }
  }
  /* first pass: counts */
  int64_t items = 0, combines = 0, prow = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t q = q_seqlens ? q_seqlens[b] : 1;
    const int64_t R = G * q;
    const int64_t QT = cdiv(R, TR);
    const int64_t NB = cdiv(context_lens[b], block_size);
    const int64_t S = cdiv(NB, c);
    items += kv_heads * QT * S;
    if (S > 1) {
      combines += kv_heads * QT;
      for (int64_t qt = 0; qt < QT; ++qt) {
        const int64_t rows = (R < (qt + 1) * TR ? R : (qt + 1) * TR) - qt * TR;
        prow += kv_heads * S * rows;
      }
    }
  }
  if (n_items) *n_items = items;
  if (n_comb) *n_comb = combines;
  if (n_partial_rows) *n_partial_rows = prow;
  if ((work && work_cap < items) || (comb && comb_cap < combines)) return 1;
  /* second pass: the lists */
  int64_t it = 0, ce = 0, slot = 0, qs = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t q = q_seqlens ? q_seqlens[b] : 1;
    const int64_t R = G * q;
    const int64_t QT = cdiv(R, TR);
    const int64_t NB = cdiv(context_lens[b], block_size);
    const int64_t S = cdiv(NB, c);
    for (int64_t kvh = 0; kvh < kv_heads; ++kvh) {
      for (int64_t qt = 0; qt < QT; ++qt) {
        const int64_t r0 = qt * TR;
        const int64_t r1 = R < r0 + TR ? R : r0 + TR;
        if (S > 1 && comb) {
          int32_t* e = comb + ce * 4;
          e[0] = b;
          e[1] = (int32_t)kvh;
          e[2] = (int32_t)it;
          e[3] = (int32_t)S;
        }
        if (S > 1) ++ce;
        for (int64_t s = 0; s < S; ++s) {
          if (work) {
            int32_t* w = work + it * 8;
            w[0] = b;
            w[1] = (int32_t)kvh;
            w[2] = (int32_t)r0;
            w[3] = (int32_t)r1;
            w[4] = (int32_t)(s * c);
            w[5] = (int32_t)(NB < (s + 1) * c ? NB : (s + 1) * c);
            w[6] = (int32_t)qs;
            w[7] = S > 1 ? (int32_t)slot : -1;
          }
          if (S > 1) slot += r1 - r0;
          ++it;
        }
      }
    }
    qs += q;
  }
  return 0;
}
