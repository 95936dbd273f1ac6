// Device-side planner: builds on the GPU, from device-resident context and
// query lengths, the same work and combine lists pa_plan builds on the host
// (the task list of SparseAttnSharedkvMetadata, "功能说明" / `metadata`, under
// the tiling and chunk rule stated in pa.h). With it a whole decode step --
// plan, attention, combine -- is a fixed sequence of launches whose sizes do
// not depend on the lengths, so it can be recorded once and replayed.
//
// One CTA of 1024 threads; thread t owns sequences 2t and 2t + 1 through the
// counting passes (their lengths stay in registers), the per-sequence counts
// are turned into offsets by one block-wide scan, and every thread then writes
// items and combine entries, finding its sequence by binary search over the
// offsets. Per-sequence arithmetic is 32-bit (lengths are int32 and checked);
// totals are 64-bit and checked against int32.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa.h"
#include "pa_internal.h"
#include "pa_plan_device.h"

namespace pa {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPerThread = 2;  // sequences a thread owns
static_assert(kPlanThreads * kPerThread >= PA_MAX_BATCH, "every sequence has an owner");

__device__ __forceinline__ int cdiv32(int a, int b) { return a / b + (a % b != 0); }

// Query rows G * q of a sequence. A launch whose total query tokens times
// heads passes INT32_MAX is rejected (as pa_plan rejects it), and G * q is at
// most that; the clamp only keeps the arithmetic of such a launch defined
// until the rejection.
__device__ __forceinline__ int rows_of(int G, int q) {
  const int64_t r = int64_t(G) * q;
  return int(r < INT32_MAX ? r : INT32_MAX);
}

// Sum of v over the CTA (all threads call it; the result is the CTA's).
__device__ int64_t block_sum64(int64_t v, int64_t* red) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int64_t t = lane < kPlanThreads / 32 ? red[lane] : 0;
  for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
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
  constexpr int kV = 4;  // counts per sequence: items, combine entries, partial rows, query tokens
  __shared__ int32_t off[kV][PA_MAX_BATCH + 1];  // exclusive offsets, off[.][B] the totals
  __shared__ int32_t nb_s[PA_MAX_BATCH];         // KV blocks of each sequence
  __shared__ int64_t red[kPlanThreads / 32];
  __shared__ int64_t wsum[kPlanThreads / 32][kV];  // warp totals, then their exclusive offsets
  __shared__ int64_t tot[kV];
  __shared__ int err, chunk_s, max_nb_s;
  __shared__ int64_t cost_s[kPlanThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = D.batch, Hk = D.kv_heads, G = D.group, bs = D.block_size, TR = D.tr;
  if (tid == 0) {
    err = 0;
    max_nb_s = 0;
  }
  __syncthreads();

  // pass 0: this thread's sequences, their checks and the work measure of the
  // automatic chunk rule
  int Ls[kPerThread], qs[kPerThread];
  int64_t w = 0;
  int mnb = 0;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int b = kPerThread * tid + k;
    Ls[k] = 1;
    qs[k] = 1;
    if (b >= B) continue;
    const int L = D.context_lens[b];
    const int q = D.q_seqlens ? D.q_seqlens[b] : 1;
    Ls[k] = L;
    qs[k] = q;
    if (q < 1 || q > D.maxq || L < q) {
      atomicOr(&err, 1);
      continue;
    }
    const int NB = cdiv32(L, bs);
    if (NB > D.max_blocks_per_seq) {
      atomicOr(&err, 1);
      continue;
    }
    w += int64_t(NB) * Hk * cdiv32(rows_of(G, q), TR);
    mnb = NB > mnb ? NB : mnb;
  }
  if (mnb) atomicMax(&max_nb_s, mnb);
  const int64_t W = block_sum64(w, red);
  if (tid == 0) {
    int64_t c = D.chunk_blocks;
    if (c <= 0) {
      c = (W + (TR <= PA_FMA_MAX_ROWS ? 8 : 2) * int64_t(D.num_sms) - 1) /
          ((TR <= PA_FMA_MAX_ROWS ? 8 : 2) * int64_t(D.num_sms));
      const int64_t RT = TR < int64_t(G) * D.maxq ? TR : int64_t(G) * D.maxq;  // real rows
      const int64_t den = int64_t(bs) * (D.hk + D.hv);
      const int64_t lo = (int64_t(64) * RT * D.hv + den - 1) / den;
      if (lo > c) c = lo;
      if (c < 1) c = 1;
    }
    chunk_s = int(c < INT32_MAX ? c : INT32_MAX);
  }
  __syncthreads();
  if (D.chunk_blocks <= 0 && TR > PA_FMA_MAX_ROWS && err == 0) {
    // wave fit (one CTA per SM): warp j prices the chunk c0 + j as its
    // waves x chunk; thread 0 takes the least, the first on a tie
    const int64_t c0 = chunk_s, cc64 = c0 + warp;
    const bool cand = cc64 <= wave_fit_hi(c0, max_nb_s);
    const int cc = int(cand ? cc64 : 1);
    int64_t n = 0;
    if (cand) {
      for (int b = lane; b < B; b += 32) {
        const int L = D.context_lens[b];
        const int q = D.q_seqlens ? D.q_seqlens[b] : 1;
        n += int64_t(Hk) * cdiv32(rows_of(G, q), TR) * cdiv32(cdiv32(L, bs), cc);
      }
    }
    for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    if (lane == 0) cost_s[warp] = cand ? (n + D.num_sms - 1) / D.num_sms * cc64 : -1;
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
  const int c = chunk_s;

  // pass 1: per-sequence counts, then their exclusive offsets by one scan
  // over the CTA (warp scans, a scan of the warp totals, the two added)
  int64_t v[kPerThread][kV], incl[kV];
#pragma unroll
  for (int j = 0; j < kV; ++j) incl[j] = 0;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int b = kPerThread * tid + k;
    const int L = Ls[k] > 0 ? Ls[k] : 1, q = qs[k] > 0 ? qs[k] : 1;
    const int NB = cdiv32(L, bs), R = rows_of(G, q), QT = cdiv32(R, TR), S = cdiv32(NB, c);
    const bool on = b < B && err == 0;
    if (b < B) nb_s[b] = NB;
    v[k][0] = on ? int64_t(Hk) * QT * S : 0;
    v[k][1] = on && S > 1 ? int64_t(Hk) * QT : 0;
    v[k][2] = on && S > 1 ? int64_t(Hk) * S * R : 0;
    v[k][3] = on ? q : 0;
#pragma unroll
    for (int j = 0; j < kV; ++j) incl[j] += v[k][j];
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int j = 0; j < kV; ++j) {
      const int64_t t = __shfl_up_sync(0xffffffffu, incl[j], o);
      if (lane >= o) incl[j] += t;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int j = 0; j < kV; ++j) wsum[warp][j] = incl[j];
  }
  __syncthreads();
  if (warp == 0) {
    int64_t x[kV], e[kV];
#pragma unroll
    for (int j = 0; j < kV; ++j) x[j] = e[j] = wsum[lane][j];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int j = 0; j < kV; ++j) {
        const int64_t t = __shfl_up_sync(0xffffffffu, e[j], o);
        if (lane >= o) e[j] += t;
      }
    }
#pragma unroll
    for (int j = 0; j < kV; ++j) {
      wsum[lane][j] = e[j] - x[j];  // exclusive offset of warp `lane`
      if (lane == 31) tot[j] = e[j];
    }
  }
  __syncthreads();
  if (tid == 0) {
    if (tot[0] > INT32_MAX || tot[2] > INT32_MAX || tot[3] * D.num_heads > INT32_MAX) err |= 1;
  }
#pragma unroll
  for (int j = 0; j < kV; ++j) {
    // exclusive offset of this thread's first sequence
    int64_t base = wsum[warp][j] + incl[j] - (v[0][j] + v[1][j]);
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const int b = kPerThread * tid + k;
      if (b < B) off[j][b] = int32_t(base < INT32_MAX ? base : INT32_MAX);
      base += v[k][j];
    }
  }
  if (tid == 0) {
#pragma unroll
    for (int j = 0; j < kV; ++j) off[j][B] = int32_t(tot[j] < INT32_MAX ? tot[j] : INT32_MAX);
  }
  __syncthreads();
  const int32_t* off_it = off[0];
  const int32_t* off_cb = off[1];
  const int32_t* off_pr = off[2];
  const int32_t* off_q = off[3];
  const int32_t N_it = off_it[B], N_cb = off_cb[B];
  const bool fail = err != 0;
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

  // the lists, in (b, kvh, qt, split) order, from shared memory alone (a
  // sequence's query tokens are the difference of its offsets); an item is
  // two 16-byte stores, a combine entry one
  for (int x = tid; x < N_it; x += kPlanThreads) {
    const int b = find_owner(off_it, B, x);
    const int q = off_q[b + 1] - off_q[b];
    const int NB = nb_s[b], R = rows_of(G, q), QT = cdiv32(R, TR), S = cdiv32(NB, c);
    const int local = x - off_it[b];
    const int kvh = local / (QT * S), rem = local % (QT * S);
    const int qt = rem / S, s = rem % S;
    const int r0 = qt * TR, r1 = R < r0 + TR ? R : r0 + TR;
    // partial rows of sequence b run (kvh, qt, s) in order: S * R per kv
    // head, S * TR per full row tile before qt, then this tile's rows per split
    const int slot = S > 1 ? off_pr[b] + kvh * S * R + qt * TR * S + s * (r1 - r0) : -1;
    int4* e = reinterpret_cast<int4*>(D.work + int64_t(x) * PA_WORK_INTS);
    e[0] = make_int4(b, kvh, r0, r1);
    e[1] = make_int4(s * c, NB < (s + 1) * c ? NB : (s + 1) * c, off_q[b], slot);
  }
  for (int y = tid; y < N_cb; y += kPlanThreads) {
    const int b = find_owner(off_cb, B, y);
    const int q = off_q[b + 1] - off_q[b];
    const int NB = nb_s[b], QT = cdiv32(rows_of(G, q), TR), S = cdiv32(NB, c);
    const int local = y - off_cb[b];
    const int kvh = local / QT, qt = local % QT;
    *reinterpret_cast<int4*>(D.combine + int64_t(y) * PA_COMBINE_INTS) =
        make_int4(b, kvh, off_it[b] + (kvh * QT + qt) * S, S);
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
