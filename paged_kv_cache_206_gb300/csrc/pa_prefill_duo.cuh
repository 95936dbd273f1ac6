// Paged attention for 256-row tiles with 128-dim heads (prefill, q = L, and
// any launch whose group rows G * max_q exceed 128) on a pair of SMs: the
// tcgen05 MMAs of cta_group::2 (M = 256) span a cluster of two CTAs, CTA c
// holding query rows 128 c .. 128 c + 127 of the work item. Same operation,
// work item and split/merge contract as the other kernels
// (PagedAttentionOperation semantics; task list and FlashDecode merge of the
// SparseAttnSharedkvMetadata page).
//
// Each CTA stages half of every operand the pair reads: 64 of a key tile's
// 128 tokens (the pair's S = Q . K^T has N = 128 tokens split between the
// two CTAs) and 64 of V's 128 dims (O += P . V has N = 128 dims, split the
// same way). A pair therefore moves each K and V byte once, and each SM's
// tensor core reads half of the B operand from its own shared memory, half
// from its peer's.
//
// Warps of each CTA (12):
//   0, 2   TMA producers of K and of V (lane 0) into this CTA's rings,
//          completing on this CTA's own landing barriers.
//   3      relays (lane 0 for K, lane 1 for V): once a slot of this CTA has
//          landed (and V rows past the item's range are zeroed), arrive on
//          CTA 0's full barrier of that slot, which thus completes when both
//          halves are in.
//   1      allocates TMEM (both CTAs, cta_group::2); in CTA 0 one thread
//          issues S(n) = Q . K(n)^T into S buffer n & 1 and O_g += P(n) . V(n)
//          (A = P from TMEM) as their inputs become ready, and commits each
//          to the barriers of both CTAs (multicast).
//   4-11   softmax in two groups that take alternate key tiles, each with its
//          own running max, sum and O accumulator (TMEM columns 256 + 128 g),
//          merged per row at the end; one row per thread. Each group arrives
//          on CTA 0's barriers when its P is written.
// A key tile wholly past one CTA's rows' causal range gets P = 0 for those
// rows (the mask's fill would give exactly zero weight). Every wait is
// bounded; on a timeout the pair records PA_STATUS_BIT_TIMEOUT and exits
// cleanly.
#pragma once

#include "pa_prefill_tc.cuh"

namespace pa {

constexpr int kDuoThreads = 384;
constexpr int kDuoRows = 128;     // query rows of one CTA (its TMEM lanes)
constexpr int kDuoKTok = 64;      // tokens of a key tile in one CTA's K slot
constexpr int kDuoSlots = 5;      // K and V slots per CTA

struct DuoCfg {
  static constexpr int HD = 128;
  static constexpr uint32_t kQ = uint32_t(kDuoRows) * HD * 2;        // 32 KB
  static constexpr uint32_t kKSlot = uint32_t(kDuoKTok) * HD * 2;    // 16 KB: [2 halves][64 tok][128 B]
  static constexpr uint32_t kVSlot = uint32_t(kPfTok) * 64 * 2;      // 16 KB: [128 tok][128 B]
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t v_off = q_off + kQ;
  static constexpr uint32_t k_off = v_off + kDuoSlots * kVSlot;
  // 16 KB after the K ring that nothing uses: every operand read the pair's
  // descriptors could make stays inside this CTA's allocation
  static constexpr uint32_t guard_off = k_off + kDuoSlots * kKSlot;
  static constexpr uint32_t bars_off = guard_off + 16384;
  static constexpr int kBars = 6 * kDuoSlots + 16;
  static constexpr uint32_t xchg_off = bars_off + kBars * 8;  // [2 groups][2][rows] fp32
  static constexpr uint32_t tmem_slot_off = xchg_off + 4 * kDuoRows * 4;
  static constexpr uint32_t bytes = tmem_slot_off + 16 + 1024;
  static_assert(bytes <= kTcMaxSmem, "shared memory");
  static_assert(v_off % 1024 == 0 && k_off % 1024 == 0, "128-byte swizzle atoms");
};

// ---- cluster primitives ----------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs of the pair.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// The address of `bar`'s twin in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}

// Arrive (release at cluster scope) on a barrier given by its cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr)
               : "memory");
}

// One poll (acquire at cluster scope) of this CTA's barrier.
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity,
                                             long long limit = kWaitLimitCycles) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_cl(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// Lane 0 waits; the whole warp gets its verdict.
__device__ __forceinline__ bool warp_wait_cl(uint64_t* bar, uint32_t parity, int lane) {
  bool ok = true;
  if (lane == 0) ok = mbar_wait_cl(bar, parity);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// D (TMEM of both CTAs) += A . B over the pair: A and B from shared memory
// (the same offsets in both CTAs: each holds its rows of A and its half of B).
__device__ __forceinline__ void tc2_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// The same with A from TMEM (each CTA's rows in its own lanes).
__device__ __forceinline__ void tc2_mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

// Arrive once on `bar` of both CTAs when every previously issued tcgen05 op of
// this thread is done.
__device__ __forceinline__ void tc2_commit_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(uint16_t(3))
      : "memory");
}

__global__ void __launch_bounds__(kDuoThreads, 1) pf_duo_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
    const FwdParams P) {
  using Cfg = DuoCfg;
  constexpr int HD = Cfg::HD;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdescQK = mma_idesc(2 * kDuoRows, kPfTok, 0, 0);
  constexpr uint32_t kIdescPV = mma_idesc(2 * kDuoRows, HD, 0, 1);
  constexpr uint32_t kHalfK = uint32_t(kDuoKTok) * 128;  // one 64-dim half of a K slot
  constexpr uint32_t kHalfQ = uint32_t(kDuoRows) * 128;  // one 64-dim half of Q
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_ctarank();  // 0 or 1: this CTA's query rows
  const bool lead = crank == 0;
  uint8_t* q_s = smem + Cfg::q_off;
  uint8_t* vring = smem + Cfg::v_off;
  uint8_t* kring = smem + Cfg::k_off;
  uint64_t* kland = reinterpret_cast<uint64_t*>(smem + Cfg::bars_off);  // this CTA's K copies landed
  uint64_t* vland = kland + kDuoSlots;   // this CTA's V copies landed (and tail zeroed)
  uint64_t* kfull = vland + kDuoSlots;   // CTA 0: both CTAs' K halves in (two relay arrivals)
  uint64_t* vfull = kfull + kDuoSlots;   // CTA 0: both V halves in
  uint64_t* kempty = vfull + kDuoSlots;  // both CTAs: the slot's QK is done (multicast commit)
  uint64_t* vempty = kempty + kDuoSlots; // both CTAs: the slot's PV is done
  uint64_t* s_full = vempty + kDuoSlots;  // [2] both CTAs: S buffer written
  uint64_t* s_free = s_full + 2;          // [2] CTA 0: S buffer read (both CTAs, 8 warps)
  uint64_t* p_full = s_full + 4;          // [2] CTA 0: P written, O rescaled (8 warps)
  uint64_t* pv_done = s_full + 6;         // [2] both CTAs: PV that read P buffer b complete
  uint64_t* qk_done = s_full + 8;
  uint64_t* o_done = s_full + 9;
  uint64_t* q_ready = s_full + 10;        // CTA 0: both query tiles in (8 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::tmem_slot_off);

  // both CTAs of a pair take the same item, so every exit below is the pair's
  const int pair = int(blockIdx.x) >> 1;
  if (P.counts && pair >= P.counts[0]) return;  // past a device plan's items
  // Items run last to first: the later row tiles of a causal sequence meet
  // more keys, so the longest items start first.
  const int n_items = P.counts ? P.counts[0] : int(gridDim.x >> 1);
  Item it;
  it.load(P, n_items - 1 - pair);
  const int G = P.group, bs = P.block_size;
  const int prefix = it.L - it.qlen;
  // key tiles each CTA's rows meet (with the compressed causal mask, up to
  // its last row's position); the pair runs the longer range
  int nt[2];
  int tok1 = it.tok0;
  for (int c = 0; c < 2; ++c) {
    const int rows = min(kDuoRows, it.nrows - c * kDuoRows);
    int t1 = it.tok0;
    if (rows > 0) {
      t1 = it.tok1;
      if (P.mask_type == PA_MASK_NORM_COMPRESS) {
        const int pmax = prefix + (it.r0 + c * kDuoRows + rows - 1) / G;
        t1 = max(it.tok0, min(it.tok1, pmax + 1));
      }
    }
    nt[c] = t1 > it.tok0 ? (t1 - it.tok0 + kPfTok - 1) / kPfTok : 0;
    tok1 = max(tok1, t1);
  }
  it.tok1 = tok1;
  const int ntiles = max(nt[0], nt[1]);
  const int nt_mine = nt[crank];
  const int sigma = it.L > PA_COMPRESS_MASK_SIZE ? it.L - PA_COMPRESS_MASK_SIZE : 0;

  if (tid == 0) {
    for (int s = 0; s < kDuoSlots; ++s) {
      mbar_init(&kland[s], 1);
      mbar_init(&vland[s], 1);
      mbar_init(&kfull[s], 2);
      mbar_init(&vfull[s], 2);
      mbar_init(&kempty[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 8);
      mbar_init(&p_full[b], 8);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(qk_done, 1);
    mbar_init(o_done, 1);
    mbar_init(q_ready, 8);
    fence_barrier_init();
  }
  // every barrier of the pair initialised before either CTA signals the other's
  cluster_sync_all();
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' TMEM allocated, the address published
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem;        // S buffer b: columns [128 b, 128 b + 128)
  const uint32_t tmem_o = tmem + 256;  // O of group g: columns [256 + 128 g, 256 + 128 g + HD)

  if (warp == 0 || warp == 2) {
    // ================= TMA producers (lane 0): K (warp 0), V (warp 2) =========
    if (lane == 0) {
      const bool is_k = warp == 0;
      const uint64_t pol = policy_evict_last();  // every row tile of the sequence reads it
      const int32_t* bt_row = P.block_tables + int64_t(it.b) * P.max_blocks_per_seq;
      // K: this CTA's 64 tokens of the tile, both 64-dim halves; V: all 128
      // tokens, this CTA's 64-dim half. Boxes of the largest power of two
      // dividing the block and the run, so that no box crosses a block.
      const int run = is_k ? kDuoKTok : kPfTok;
      const int box_rows = (bs & -bs) < run ? (bs & -bs) : run;
      const int pieces = run / box_rows;
      const int tok_off = is_k ? int(crank) * kDuoKTok : 0;
      const int z0 = is_k ? it.kvh * (HD / 64) : it.kvh * ((P.kv_shared ? P.hk : HD) / 64) + int(crank);
      const uint32_t piece_bytes = uint32_t(box_rows) * 128 * (is_k ? 2 : 1);
      uint64_t* landb = is_k ? kland : vland;
      uint64_t* emptyb = is_k ? kempty : vempty;
      uint8_t* ring = is_k ? kring : vring;
      const uint32_t slot_bytes = is_k ? Cfg::kKSlot : Cfg::kVSlot;
      const CUtensorMap* map = is_k ? &tmk : &tmv;
      int iss = 0;
      bool ok = true;
      for (int n = 0; n < ntiles; ++n) {
        const int t0 = it.tok0 + n * kPfTok + tok_off;
        int npieces = 0;
        for (int pc = 0; pc < pieces; ++pc) {
          const int tok = t0 + pc * box_rows;
          if (tok >= it.tok1) break;
          const int ph = bt_row[tok / bs];
          if (ph < 0 || ph >= P.num_blocks) {
            if (is_k) set_status(P.status, PA_STATUS_BIT_BLOCK_INDEX);
            continue;
          }
          ++npieces;
        }
        const int slot = iss % kDuoSlots;
        if (!mbar_wait(&emptyb[slot], ((iss / kDuoSlots) & 1) ^ 1)) {
          ok = false;
          break;
        }
        uint8_t* dst = ring + slot * slot_bytes;
        uint64_t* land = &landb[slot];
        const uint32_t bytes = uint32_t(npieces) * piece_bytes;
        if (bytes) mbar_arrive_expect_tx(land, bytes); else mbar_arrive(land);
        for (int pc = 0; pc < pieces; ++pc) {
          const int tok = t0 + pc * box_rows;
          if (tok >= it.tok1) break;
          const int ph = bt_row[tok / bs];
          if (ph < 0 || ph >= P.num_blocks) continue;
          const int row = ph * bs + tok % bs;
          if (is_k && box_rows == kDuoKTok) {
            tma_load_3d(dst, map, land, 0, row, z0, pol);  // [2 halves][64 tokens][128 B]
          } else if (is_k) {
            for (int h = 0; h < 2; ++h)
              tma_load_3d(dst + h * kHalfK + pc * box_rows * 128, map, land, 0, row, z0 + h, pol);
          } else {
            tma_load_3d(dst + pc * box_rows * 128, map, land, 0, row, z0, pol);  // [rows][128 B]
          }
        }
        ++iss;
      }
      if (!ok) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
      for (int i = iss - kDuoSlots > 0 ? iss - kDuoSlots : 0; i < iss; ++i)
        mbar_wait(&landb[i % kDuoSlots], (i / kDuoSlots) & 1);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ================= relays: K (lane 0), V (lane 1) =================
    // This CTA's half of K(n) or V(n) landed (V rows past the item's range
    // zeroed: they may hold anything, NaN included, and P = 0 there): tell
    // CTA 0's MMA thread. Separate lanes, so that a late V tile never holds
    // back the next QK.
    if (lane < 2) {
      const bool is_k = lane == 0;
      uint64_t* landb = is_k ? kland : vland;
      uint64_t* fullb = is_k ? kfull : vfull;
      bool ok = true;
      for (int n = 0; n < ntiles; ++n) {
        const int s = n % kDuoSlots;
        if (!mbar_wait(&landb[s], (n / kDuoSlots) & 1)) { ok = false; break; }
        const int nvalid = min(kPfTok, it.tok1 - (it.tok0 + n * kPfTok));
        if (!is_k && nvalid < kPfTok) {
          uint8_t* vb = vring + s * Cfg::kVSlot;
          for (int idx = nvalid * 8; idx < kPfTok * 8; ++idx)
            *reinterpret_cast<uint4*>(vb + idx * 16) = make_uint4(0, 0, 0, 0);
          fence_proxy_async();  // written by this thread, read by the tensor cores
        }
        mbar_arrive_cluster(peer_addr(&fullb[s], 0));
      }
      if (!ok) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer (CTA 0) =================
    // S(n) into buffer n & 1 and O_g += P(n) V(n) in whatever order their
    // inputs become ready; lane 0 polls, the warp follows its verdicts.
    if (lead) {
      bool ok = true;
      const uint32_t q_addr = smem_u32(q_s);
      const uint32_t k_addr = smem_u32(kring), v_addr = smem_u32(vring);
      if (ntiles > 0 && !warp_wait_cl(q_ready, 0, lane)) ok = false;
      auto ready = [&](uint64_t* bar, uint32_t parity) -> bool {
        const bool r = lane == 0 ? mbar_try_wait_cl(bar, parity) : false;
        return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
      };
      int nq = 0, np = 0;  // next QK tile, next PV tile
      long long idle_since = clock64();
      while (ok && np < ntiles) {
        bool progressed = false;
        // QK(nq): both K halves are in, and its S buffer's P (tile nq - 2) was
        // read by PV(nq - 2), issued before it by this thread (the tensor
        // cores carry one thread's MMAs out in order)
        if (nq < ntiles && (nq < 2 || (np >= nq - 1 && ready(&s_free[nq & 1], ((nq >> 1) - 1) & 1))) &&
            ready(&kfull[nq % kDuoSlots], (nq / kDuoSlots) & 1)) {
          const int ks = nq % kDuoSlots;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int h = 0; h < HD / 64; ++h) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t a = smem_desc(q_addr + h * kHalfQ + k * 32, 16, 1024);
                const uint64_t b = smem_desc(k_addr + ks * Cfg::kKSlot + h * kHalfK + k * 32, 16, 1024);
                tc2_mma(tmem_s + (nq & 1) * 128, a, b, kIdescQK, (h | k) != 0);
              }
            }
            tc2_commit_both(&kempty[ks]);
            tc2_commit_both(&s_full[nq & 1]);
          }
          __syncwarp();
          ++nq;
          progressed = true;
        }
        // PV(np): both CTAs' P written, both V halves in
        if (np < nq && ready(&p_full[np & 1], (np >> 1) & 1) &&
            ready(&vfull[np % kDuoSlots], (np / kDuoSlots) & 1)) {
          const int m = np, pb = m & 1, vs = m % kDuoSlots;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kPfTok / 16; ++k) {
              // A = P in TMEM (16 tokens = 8 columns of fp16 pairs); B = this
              // CTA's 64 dims of V (tokens x dims, MN-major, one 64-dim block)
              const uint64_t b = smem_desc(v_addr + vs * Cfg::kVSlot + k * 2048, Cfg::kVSlot, 1024);
              tc2_mma_tmem_a(tmem_o + pb * 128, tmem_s + pb * 128 + k * 8, b, kIdescPV,
                             ((m >> 1) | k) != 0);
            }
            tc2_commit_both(&vempty[vs]);
            tc2_commit_both(&pv_done[pb]);
          }
          __syncwarp();
          ++np;
          progressed = true;
        }
        if (progressed) {
          idle_since = clock64();
        } else if (clock64() - idle_since > kWaitLimitCycles) {
          ok = false;  // nothing became ready within the wait limit
        }
      }
      if (!ok && lane == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
      if (lane == 0) {
        tc2_commit_both(qk_done);
        tc2_commit_both(o_done);
      }
      __syncwarp();
    }
  } else {
    // ================= softmax: group g (warps 4-7 / 8-11) takes tiles n = g mod 2 =====
    const int grp = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                // TMEM lane = row of this CTA's tile
    const int ri = int(crank) * kDuoRows + r;         // row of the item
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const bool row_ok = ri < it.nrows;
    const int rr = it.r0 + ri;
    const int qi = row_ok ? rr / G : 0;  // query token of the row
    const int p_row = prefix + qi;       // its position
    const float slope = (row_ok && P.mask_type == PA_MASK_ALIBI)
                            ? P.alibi_slopes[it.kvh * G + rr % G] * kLog2e : 0.f;
    const uint32_t q_ready_cl = peer_addr(q_ready, 0);
    if (grp == 0) {
      // this CTA's query rows: 64-dim halves, swizzled; 128 threads, 16-byte chunks
      const int st = tid - 128;
      constexpr int kChunks = kDuoRows * (HD / 8);
      constexpr int kPer = kChunks / 128, kRound = kPer < 8 ? kPer : 8;
#pragma unroll
      for (int k0 = 0; k0 < kPer; k0 += kRound) {
        uint4 v[kRound];  // every load of the round before any store
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
          const int idx = st + (k0 + k) * 128;
          const int row = idx / (HD / 8), c = idx % (HD / 8);
          v[k] = make_uint4(0, 0, 0, 0);
          if (int(crank) * kDuoRows + row < it.nrows) {
            const int rq = it.r0 + int(crank) * kDuoRows + row;
            v[k] = *reinterpret_cast<const uint4*>(
                P.query + (int64_t(it.q_start + rq / G) * P.num_heads + it.kvh * G + rq % G) * HD + c * 8);
          }
        }
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
          const int idx = st + (k0 + k) * 128;
          const int row = idx / (HD / 8), c = idx % (HD / 8);
          *reinterpret_cast<uint4*>(q_s + (c >> 3) * kHalfQ + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = v[k];
        }
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(q_ready_cl);
    }
    const uint32_t s_free_cl[2] = {peer_addr(&s_free[0], 0), peer_addr(&s_free[1], 0)};
    const uint32_t p_full_cl[2] = {peer_addr(&p_full[0], 0), peer_addr(&p_full[1], 0)};
    float m_ref = -INFINITY;  // reference max of the row over this group's tiles (base 2)
    float l = 0.f;            // sum of exp2(s - m_ref) over those keys
    bool ok = true;
    for (int n = grp; n < ntiles; n += 2) {
      const int b = n & 1;  // = grp: S, P and O buffers of this group
      if (!warp_wait_cl(&s_full[b], (n >> 1) & 1, lane)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sbuf = tmem_s + b * 128 + lane_base;
      const uint32_t o_mine = tmem_o + b * 128 + lane_base;
      if (n >= nt_mine) {
        // a tile past every row's causal range in this CTA: P = 0, no state
        // change (the mask's fill would give exactly zero weight). The P
        // rewrite still waits for this group's previous PV.
        if (n >= 2 && !__all_sync(0xffffffffu, mbar_wait_cl(&pv_done[b], ((n - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
        for (int cc = 0; cc < kPfTok / 32; ++cc) tmem_st16u(sbuf + cc * 16, z);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_cluster(s_free_cl[b]);
          mbar_arrive_cluster(p_full_cl[b]);
        }
        continue;
      }
      // Pass 1, 32 columns at a time: scores in base 2 with the bias, written
      // back into the S buffer, and the tile's row max.
      const int j0 = it.tok0 + n * kPfTok;  // key of column 0
      const int jend = it.tok1 - j0;       // columns at or past this are outside the range
      float tmax = -INFINITY;
      // (tcgen05.ld / st are warp-collective: the branch below must be taken by
      // the whole warp, so the test is whether any row of the warp needs it)
      const bool diag_row = row_ok && j0 + kPfTok - 1 > p_row;
      if (P.mask_type == PA_MASK_NORM_COMPRESS && __any_sync(0xffffffffu, diag_row)) {
        const int mr = min(max(p_row - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
        const __half* mrow = P.mask + mr * PA_COMPRESS_MASK_SIZE;
#pragma unroll 1
        for (int cc = 0; cc < kPfTok / 32; ++cc) {
          float x[32];
          tmem_ld32(sbuf + cc * 32, x);
          const bool need = __any_sync(0xffffffffu, diag_row && j0 + cc * 32 + 31 > p_row);
          __half mv[32];
          if (need) {
            const int m0 = j0 + cc * 32 - sigma;  // mask column of this chunk's first key
            if (m0 >= 0 && m0 + 32 <= PA_COMPRESS_MASK_SIZE && (m0 & 7) == 0) {
              const uint4* src = reinterpret_cast<const uint4*>(mrow + m0);
#pragma unroll
              for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(mv + 8 * q) = src[q];
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                mv[i] = mrow[min(max(m0 + i, 0), PA_COMPRESS_MASK_SIZE - 1)];
            }
          }
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c = cc * 32 + i, j = j0 + c;
            float v = x[i] * P.scale_log2;
            if (need && diag_row && j > p_row && c < jend) v += __half2float(mv[i]) * kLog2e;
            v = c < jend ? v : -INFINITY;
            x[i] = v;
            tmax = fmaxf(tmax, v);
          }
          tmem_st32(sbuf + cc * 32, x);
        }
      } else if (P.mask_type == PA_MASK_ALIBI || P.mask_type == PA_MASK_NORM) {
        const bool alibi = P.mask_type == PA_MASK_ALIBI;
#pragma unroll 1
        for (int cc = 0; cc < kPfTok / 32; ++cc) {
          float x[32];
          tmem_ld32(sbuf + cc * 32, x);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c = cc * 32 + i, j = j0 + c;
            float v = x[i] * P.scale_log2;
            if (alibi) v += slope * float(j - p_row);
            else if (row_ok && c < jend) v += norm_mask_log2(P, it.b, qi, j);
            v = c < jend ? v : -INFINITY;
            x[i] = v;
            tmax = fmaxf(tmax, v);
          }
          tmem_st32(sbuf + cc * 32, x);
        }
      } else {
#pragma unroll 1
        for (int cc = 0; cc < kPfTok / 32; ++cc) {
          float x[32];
          tmem_ld32(sbuf + cc * 32, x);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float v = cc * 32 + i < jend ? x[i] * P.scale_log2 : -INFINITY;
            x[i] = v;
            tmax = fmaxf(tmax, v);
          }
          tmem_st32(sbuf + cc * 32, x);
        }
      }
      tmem_wait_st();
      // move the reference only when a score passes it by more than 2^8
      const bool grow = tmax > m_ref + kTcRescaleThreshold;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m_ref - tmax);  // 0 on this group's first tile
        m_ref = tmax;
        l *= alpha;
      }
      // this group's previous PV (tile n - 2) read P buffer b and wrote O: both
      // the P rewrite and a rescale of O wait for it
      if (n >= 2 && !__all_sync(0xffffffffu, mbar_wait_cl(&pv_done[b], ((n - 2) >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Pass 2: probabilities as fp16 pairs into the S buffer's first 64
      // columns, where the PV MMA reads them
      float psum = 0.f;
#pragma unroll 1
      for (int cc = 0; cc < kPfTok / 32; ++cc) {
        float x[32];
        tmem_ld32(sbuf + cc * 32, x);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float e0 = ex2(x[2 * i] - m_ref), e1 = ex2(x[2 * i + 1] - m_ref);
          psum += e0 + e1;
          pk[i] = pack_half2(e0, e1);
        }
        tmem_st16u(sbuf + cc * 16, pk);
      }
      l += psum;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(s_free_cl[b]);
      if (n >= 2 && __any_sync(0xffffffffu, grow && row_ok)) {
        // rescale this warp's rows of this group's O (rows that did not grow use 1)
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          float o[32];
          tmem_ld32(o_mine + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(o_mine + c * 32, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(p_full_cl[b]);
    }
    if (!ok && lane == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    launch_dependents();
    // ---- merge the two groups' states per row; group g writes dims 64 g ..
    float* xm = reinterpret_cast<float*>(smem + Cfg::xchg_off);  // [group][m, l][rows]
    xm[(grp * 2) * kDuoRows + r] = m_ref;
    xm[(grp * 2 + 1) * kDuoRows + r] = l;
    asm volatile("bar.sync 1, 256;" ::: "memory");  // the 8 softmax warps
    const bool got = ok && warp_wait_cl(o_done, 0, lane);
    const bool partial = it.slot >= 0;
    const bool fits = !partial || int64_t(it.slot) + it.nrows <= P.part_rows_cap;
    if (!fits && ri == 0 && grp == 0) set_status(P.status, PA_STATUS_BIT_WORKSPACE);
    if (got && fits) {
      tc_fence_after();
      const bool two = ntiles >= 2;  // group 1 ran (and wrote its O)
      const float m0 = xm[r], l0 = xm[kDuoRows + r];
      const float m1 = two ? xm[2 * kDuoRows + r] : -INFINITY, l1 = two ? xm[3 * kDuoRows + r] : 0.f;
      const float mm = fmaxf(m0, m1);
      const float a0 = (ntiles > 0 && l0 > 0.f) ? ex2(m0 - mm) : 0.f;
      const float a1 = (two && l1 > 0.f) ? ex2(m1 - mm) : 0.f;
      const float lt = l0 * a0 + l1 * a1;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float w0 = a0 * inv, w1 = a1 * inv;
#pragma unroll 1
      for (int c = 2 * grp; c < 2 * grp + 2; ++c) {
        float o[32], o1[32];
        tmem_ld32(tmem_o + c * 32 + lane_base, o);
        if (two) {
          tmem_ld32(tmem_o + 128 + c * 32 + lane_base, o1);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o1[i] = 0.f;
        }
        tmem_wait_ld();
        if (!row_ok) continue;
        // a group whose weight is zero (no tile, or every key of the row
        // masked in its tiles) adds nothing, whatever its accumulator holds
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = (w0 != 0.f ? o[i] * w0 : 0.f) + (w1 != 0.f ? o1[i] * w1 : 0.f);
        if (partial) {
          float4* dst = reinterpret_cast<float4*>(P.part_o + (int64_t(it.slot) + ri) * HD + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(
              P.out + (int64_t(it.q_start + qi) * P.num_heads + it.kvh * G + rr % G) * HD + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 pk;
            pk.x = pack_half2(o[8 * i + 0], o[8 * i + 1]);
            pk.y = pack_half2(o[8 * i + 2], o[8 * i + 3]);
            pk.z = pack_half2(o[8 * i + 4], o[8 * i + 5]);
            pk.w = pack_half2(o[8 * i + 6], o[8 * i + 7]);
            dst[i] = pk;
          }
        }
      }
      if (partial && row_ok && grp == 0)
        P.part_lse[it.slot + ri] = lt > 0.f ? (mm + log2f(lt)) * kLn2 : -INFINITY;
    }
  }
  // ---- teardown: every tcgen05 op of the pair has completed (o_done, in both
  // CTAs) before either frees TMEM or leaves: the pair MMAs read both CTAs'
  // shared memory and TMEM
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    if (lane == 0) {
      mbar_wait_cl(qk_done, 0);
      mbar_wait_cl(o_done, 0);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols));
  }
  cluster_sync_all();
}

}  // namespace pa
