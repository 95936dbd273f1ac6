// Device-side planner: builds on the GPU, from device-resident context and
// query lengths, the same work and combine lists pa_plan builds on the host
// (the task list of SparseAttnSharedkvMetadata, "功能说明" / `metadata`, under
// the tiling and chunk rule stated in pa.h). With it a whole decode step --
// plan, attention, combine -- is a fixed sequence of launches whose sizes do
// not depend on the lengths, so it can be recorded once and replayed.
//
// One CTA of 1024 threads: sequence b is owned by threads b and b + 1024 of
// the first pass; per-sequence counts are prefix-summed by warp 0 (64
// sequences per lane, then a warp scan); every thread then writes items and
// combine entries, finding its sequence by binary search over the offsets.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa.h"
#include "pa_internal.h"
#include "pa_plan_device.h"

namespace pa {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPerLane = (PA_MAX_BATCH + 31) / 32;  // sequences per lane of the scan

__device__ __forceinline__ int64_t dcdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

__device__ int64_t block_sum64(int64_t v, int64_t* red) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int64_t t = 0;
  for (int w = 0; w < kPlanThreads / 32; ++w) t += red[w];
  return t;
}

// Position of key x in the non-decreasing offsets off[0..n]: the b with
// off[b] <= x < off[b + 1].
__device__ __forceinline__ int find_owner(const int32_t* off, int n, int32_t x) {
  int lo = 0, hi = n;  // off[lo] <= x < off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(const DevPlanParams D) {
  __shared__ int32_t off_it[PA_MAX_BATCH + 1];  // items before sequence b
  __shared__ int32_t off_cb[PA_MAX_BATCH + 1];  // combine entries before b
  __shared__ int32_t off_pr[PA_MAX_BATCH + 1];  // partial rows before b
  __shared__ int32_t off_q[PA_MAX_BATCH + 1];   // query tokens before b
  __shared__ int64_t red[kPlanThreads / 32];
  __shared__ int err, chunk_s, max_nb_s;
  __shared__ int64_t cost_s[kPlanThreads / 32];
  const int tid = threadIdx.x;
  const int B = D.batch, Hk = D.kv_heads, G = D.group, bs = D.block_size, TR = D.tr;
  if (tid == 0) {
    err = 0;
    max_nb_s = 0;
  }
  __syncthreads();

  // pass 0: checks and the work measure of the automatic chunk rule
  int64_t w = 0;
  int mnb = 0;
  for (int b = tid; b < B; b += kPlanThreads) {
    const int64_t L = D.context_lens[b];
    const int64_t q = D.q_seqlens ? D.q_seqlens[b] : 1;
    const int64_t NB = dcdiv(L, bs);
    if (q < 1 || q > D.maxq || L < q || NB > D.max_blocks_per_seq) {
      atomicOr(&err, 1);
      continue;
    }
    w += NB * Hk * dcdiv(G * q, TR);
    mnb = NB > mnb ? int(NB) : mnb;
  }
  atomicMax(&max_nb_s, mnb);
  const int64_t W = block_sum64(w, red);
  if (tid == 0) {
    int64_t c = D.chunk_blocks;
    if (c <= 0) {
      c = dcdiv(W, (TR <= PA_FMA_MAX_ROWS ? 8 : 2) * int64_t(D.num_sms));
      const int64_t RT = TR < int64_t(G) * D.maxq ? TR : int64_t(G) * D.maxq;  // real rows
      const int64_t lo = dcdiv(int64_t(64) * RT * D.hv, int64_t(bs) * (D.hk + D.hv));
      if (lo > c) c = lo;
      if (c < 1) c = 1;
    }
    chunk_s = int(c < INT32_MAX ? c : INT32_MAX);
  }
  __syncthreads();
  if (D.chunk_blocks <= 0 && TR > PA_FMA_MAX_ROWS) {
    // wave fit (one CTA per SM): warp j prices the chunk c0 + j as its
    // waves x chunk; thread 0 takes the least, the first on a tie
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t c0 = chunk_s, cc = c0 + warp;
    const bool cand = cc <= wave_fit_hi(c0, max_nb_s);
    int64_t n = 0;
    if (cand) {
      for (int b = lane; b < B; b += 32) {
        const int64_t L = D.context_lens[b];
        const int64_t q = D.q_seqlens ? D.q_seqlens[b] : 1;
        if (q < 1 || L < q) continue;  // reported through err
        n += int64_t(Hk) * dcdiv(int64_t(G) * q, TR) * dcdiv(dcdiv(L, bs), cc);
      }
    }
    for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    if (lane == 0) cost_s[warp] = cand ? dcdiv(n, int64_t(D.num_sms)) * cc : -1;
    __syncthreads();
    if (tid == 0) {
      int64_t best = c0, best_cost = -1;
      for (int j = 0; j < kPlanThreads / 32; ++j) {
        if (cost_s[j] < 0) continue;
        if (best_cost < 0 || cost_s[j] < best_cost) {
          best_cost = cost_s[j];
          best = c0 + j;
        }
      }
      chunk_s = int(best < INT32_MAX ? best : INT32_MAX);
    }
    __syncthreads();
  }
  const int64_t c = chunk_s;

  // pass 1: per-sequence counts (64-bit totals checked against int32)
  int64_t t_it = 0, t_pr = 0, t_q = 0;
  for (int b = tid; b < B; b += kPlanThreads) {
    const int64_t L = D.context_lens[b];
    const int64_t q = D.q_seqlens ? D.q_seqlens[b] : 1;
    const int64_t NB = dcdiv(L > 0 ? L : 1, bs);
    const int64_t R = G * q, QT = dcdiv(R, TR), S = dcdiv(NB, c);
    const int64_t items = Hk * QT * S;
    const int64_t prows = S > 1 ? Hk * S * R : 0;
    t_it += items;
    t_pr += prows;
    t_q += q;
    off_it[b] = int32_t(items < INT32_MAX ? items : INT32_MAX);
    off_cb[b] = int32_t(S > 1 ? Hk * QT : 0);
    off_pr[b] = int32_t(prows < INT32_MAX ? prows : INT32_MAX);
    off_q[b] = int32_t(q);
  }
  const int64_t n_items = block_sum64(t_it, red);
  const int64_t n_prows = block_sum64(t_pr, red);
  const int64_t n_q = block_sum64(t_q, red);
  if (tid == 0) {
    if (n_items > INT32_MAX || n_prows > INT32_MAX || n_q * D.num_heads > INT32_MAX)
      err |= 1;
  }
  __syncthreads();

  // exclusive prefix sums over the sequences (warp 0)
  if (tid < 32) {
    const int lane = tid;
    const int b0 = lane * kPerLane;
    int32_t s_it = 0, s_cb = 0, s_pr = 0, s_q = 0;
    for (int k = 0; k < kPerLane; ++k) {
      const int b = b0 + k;
      if (b < B) {
        s_it += off_it[b];
        s_cb += off_cb[b];
        s_pr += off_pr[b];
        s_q += off_q[b];
      }
    }
    int32_t e_it = s_it, e_cb = s_cb, e_pr = s_pr, e_q = s_q;  // inclusive, then exclusive
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t a = __shfl_up_sync(0xffffffffu, e_it, o);
      const int32_t bb = __shfl_up_sync(0xffffffffu, e_cb, o);
      const int32_t cc = __shfl_up_sync(0xffffffffu, e_pr, o);
      const int32_t dd = __shfl_up_sync(0xffffffffu, e_q, o);
      if (lane >= o) {
        e_it += a;
        e_cb += bb;
        e_pr += cc;
        e_q += dd;
      }
    }
    e_it -= s_it;
    e_cb -= s_cb;
    e_pr -= s_pr;
    e_q -= s_q;
    for (int k = 0; k < kPerLane; ++k) {
      const int b = b0 + k;
      if (b < B) {
        const int32_t vi = off_it[b], vc = off_cb[b], vp = off_pr[b], vq = off_q[b];
        off_it[b] = e_it;
        off_cb[b] = e_cb;
        off_pr[b] = e_pr;
        off_q[b] = e_q;
        e_it += vi;
        e_cb += vc;
        e_pr += vp;
        e_q += vq;
      }
    }
    if (lane == 31) {
      off_it[B] = e_it;
      off_cb[B] = e_cb;
      off_pr[B] = e_pr;
      off_q[B] = e_q;
    }
  }
  __syncthreads();
  const int32_t N_it = off_it[B], N_cb = off_cb[B];
  bool fail = err != 0;
  const bool small = !fail && (N_it > D.work_cap || N_cb > D.comb_cap);
  if (fail || small) {
    if (tid == 0) {
      D.counts[0] = 0;
      D.counts[1] = 0;
      D.counts[2] = 0;
      D.counts[3] = fail ? 1 : 2;
      atomicOr(D.status, fail ? PA_STATUS_BIT_PLAN : PA_STATUS_BIT_WORKSPACE);
    }
    return;
  }

  // the lists, in (b, kvh, qt, split) order
  for (int x = tid; x < N_it; x += kPlanThreads) {
    const int b = find_owner(off_it, B, x);
    const int64_t L = D.context_lens[b];
    const int64_t q = D.q_seqlens ? D.q_seqlens[b] : 1;
    const int64_t NB = dcdiv(L, bs), R = G * q, QT = dcdiv(R, TR), S = dcdiv(NB, c);
    const int64_t local = x - off_it[b];
    const int64_t kvh = local / (QT * S), rem = local % (QT * S);
    const int64_t qt = rem / S, s = rem % S;
    const int64_t r0 = qt * TR, r1 = R < r0 + TR ? R : r0 + TR;
    int32_t* e = D.work + int64_t(x) * PA_WORK_INTS;
    e[0] = b;
    e[1] = int32_t(kvh);
    e[2] = int32_t(r0);
    e[3] = int32_t(r1);
    e[4] = int32_t(s * c);
    e[5] = int32_t(NB < (s + 1) * c ? NB : (s + 1) * c);
    e[6] = off_q[b];
    // partial rows of sequence b run (kvh, qt, s) in order: S * R per kv
    // head, S * TR per full row tile before qt, then this tile's rows per split
    e[7] = S > 1 ? int32_t(off_pr[b] + kvh * S * R + qt * TR * S + s * (r1 - r0)) : -1;
  }
  for (int y = tid; y < N_cb; y += kPlanThreads) {
    const int b = find_owner(off_cb, B, y);
    const int64_t L = D.context_lens[b];
    const int64_t q = D.q_seqlens ? D.q_seqlens[b] : 1;
    const int64_t NB = dcdiv(L, bs), QT = dcdiv(G * q, TR), S = dcdiv(NB, c);
    const int64_t local = y - off_cb[b];
    const int64_t kvh = local / QT, qt = local % QT;
    int32_t* e = D.combine + int64_t(y) * PA_COMBINE_INTS;
    e[0] = b;
    e[1] = int32_t(kvh);
    e[2] = int32_t(off_it[b] + (kvh * QT + qt) * S);
    e[3] = int32_t(S);
  }
  if (tid == 0) {
    D.counts[0] = N_it;
    D.counts[1] = N_cb;
    D.counts[2] = off_pr[B];
    D.counts[3] = 0;
  }
}

}  // namespace

cudaError_t launch_plan(const DevPlanParams& D, cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(D);
  return cudaGetLastError();
}

}  // namespace pa
