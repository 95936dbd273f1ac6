// Paged attention for 128-row tiles whose rows meet many keys (launches whose
// group rows G * max_q are 65 to 128 with 64/128-dim heads: wide groups, short
// prefill; beyond 128 rows the 256-row kernel of pa_prefill_pair.cuh takes
// over), on the tcgen05 tensor cores. Same operation, work item and
// split/merge contract as the decode kernels (PagedAttentionOperation
// semantics; task list and FlashDecode merge of the SparseAttnSharedkvMetadata
// page); a different tile shape.
//
// One CTA per work item (a 128-row tile), 128-token key tiles, 12 warps:
//   warps 0, 2 TMA producers of K and of V: each key tile as 3-D boxes
//              (128-byte swizzle) into 3-slot K and V rings.
//   warp 1     allocates TMEM; one thread issues S = Q . K^T (M=128 rows,
//              N=128 tokens, K-major operands; S double-buffered in TMEM)
//              and O += P . V (M=128, N=hd; A = P from TMEM, B = V MN-major;
//              O accumulates in TMEM), each as soon as its inputs are ready.
//   warps 4-11 softmax in two groups of four that take alternate key tiles,
//              each with its own running max, sum and O accumulator (merged
//              per row at the end); one query row per thread (TMEM lane m
//              holds row m of an M=128 accumulator): the row's
//              scores come from TMEM in 32-column loads, so max and sum need
//              no exchange between threads. The reference max is moved (and
//              O rescaled in TMEM) only when a score exceeds it by more than
//              2^8. P (fp16) is written back into the S buffer's TMEM
//              columns, where the PV MMA takes it as its A operand.
//   warp 3     no role.
// With the compressed causal mask an item stops after its last query row's
// position, and only the keys above the diagonal read the mask. Every wait is
// bounded; on a timeout the CTA records PA_STATUS_BIT_TIMEOUT and exits
// cleanly.
#pragma once

#include "pa_decode_tc.cuh"

namespace pa {

constexpr int kPfTok = 128;      // key tokens per tile (N of S = Q . K^T)
constexpr int kPfRows = PA_PF_TILE_ROWS;  // query rows per tile (M of both MMAs)
constexpr int kPfThreads = 384;  // 12 warps
constexpr int kPfKSlots = 3;
constexpr int kPfVSlots = 3;

// 16 columns of 32-bit values into this warp's TMEM lane quarter.
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// D (TMEM) += A (TMEM: row m in lane m, K in consecutive 32-bit columns of
// fp16 pairs) . B (shared memory descriptor).
__device__ __forceinline__ void tc_mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

template <int HD>
struct PfCfg {
  static constexpr int kHalves = HD / 64;                       // 64-dim halves of a row
  static constexpr uint32_t kSlot = uint32_t(kPfTok) * HD * 2;  // one K or V tile
  static constexpr uint32_t kQ = uint32_t(kPfRows) * HD * 2;
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t k_off = q_off + kQ;
  static constexpr uint32_t v_off = k_off + kPfKSlots * kSlot;
  static constexpr uint32_t bars_off = v_off + kPfVSlots * kSlot;
  static constexpr int kBars = 2 * (kPfKSlots + kPfVSlots) + 12;
  static constexpr uint32_t xchg_off = bars_off + kBars * 8;  // [2][rows] fp32 row merge
  static constexpr uint32_t tmem_slot_off = xchg_off + 2 * kPfRows * 4;
  static constexpr uint32_t bytes = tmem_slot_off + 16 + 1024;
  static_assert(bytes <= kTcMaxSmem, "shared memory");
};

inline bool pf_supported(int hk, int hv) { return hk == hv && (hk == 64 || hk == 128); }

template <int HD>
__global__ void __launch_bounds__(kPfThreads, 1) pf_attn_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
    const FwdParams P) {
  using Cfg = PfCfg<HD>;
  constexpr int H2 = Cfg::kHalves;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdescQK = mma_idesc(kPfRows, kPfTok, 0, 0);
  constexpr uint32_t kIdescPV = mma_idesc(kPfRows, HD, 0, 1);
  constexpr uint32_t kHalfK = uint32_t(kPfTok) * 128;  // one 64-dim half of a K/V tile
  constexpr uint32_t kHalfQ = uint32_t(kPfRows) * 128;  // one 64-dim half of Q
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* q_s = smem + Cfg::q_off;
  uint8_t* kring = smem + Cfg::k_off;
  uint8_t* vring = smem + Cfg::v_off;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + Cfg::bars_off);
  uint64_t* kempty = kfull + kPfKSlots;
  uint64_t* vfull = kempty + kPfKSlots;
  uint64_t* vempty = vfull + kPfVSlots;
  uint64_t* s_full = vempty + kPfVSlots;  // [2] S buffer written
  uint64_t* s_free = s_full + 2;          // [2] S buffer read and P written by the softmax warps
  uint64_t* p_full = s_full + 4;          // [2] P buffer written
  uint64_t* pv_done = s_full + 6;         // [2] PV that read P buffer b complete
  uint64_t* qk_done = s_full + 8;
  uint64_t* o_done = s_full + 9;
  uint64_t* q_ready = s_full + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::tmem_slot_off);

  if (P.counts && int(blockIdx.x) >= P.counts[0]) return;  // past a device plan's items
  // Items run last to first: with the causal mask the later row tiles of a
  // sequence meet more keys, so the longest items start first and the last
  // wave holds the short ones.
  const int n_items = P.counts ? P.counts[0] : int(gridDim.x);
  Item it;
  it.load(P, n_items - 1 - int(blockIdx.x));
  const int G = P.group, bs = P.block_size;
  const int prefix = it.L - it.qlen;
  if (P.mask_type == PA_MASK_NORM_COMPRESS && it.nrows > 0) {
    // causal trim, as in the decode kernel: keys past the last row's position
    // carry the mask's fill for every row of the tile
    const int pmax = prefix + (it.r0 + it.nrows - 1) / G;
    it.tok1 = max(it.tok0, min(it.tok1, pmax + 1));
  }
  const int ntok = it.tok1 - it.tok0;
  const int ntiles = ntok > 0 ? (ntok + kPfTok - 1) / kPfTok : 0;
  const int sigma = it.L > PA_COMPRESS_MASK_SIZE ? it.L - PA_COMPRESS_MASK_SIZE : 0;

  if (tid == 0) {
    for (int s = 0; s < kPfKSlots; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < kPfVSlots; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 4);
      mbar_init(&p_full[b], 4);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(qk_done, 1);
    mbar_init(o_done, 1);
    mbar_init(q_ready, 4);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem;        // S buffer b: columns [128 b, 128 b + 128)
  const uint32_t tmem_o = tmem + 256;  // O of group g: columns [256 + 128 g, 256 + 128 g + HD)

  if (warp == 0 || warp == 2) {
    // ================= TMA producers (lane 0): K (warp 0), V (warp 2) =========
    // Separate producers, so that a K tile never waits behind a V tile whose
    // slot is still being read.
    if (lane == 0) {
      const bool is_k = warp == 0;
      const uint64_t pol = policy_evict_last();  // every row tile of the sequence reads it
      const int32_t* bt_row = P.block_tables + int64_t(it.b) * P.max_blocks_per_seq;
      // the largest power of two dividing both the block and the tile: a
      // box never crosses a block (block_size 48 moves 16-token boxes)
      const int box_rows = (bs & -bs) < kPfTok ? (bs & -bs) : kPfTok;
      const int pieces = kPfTok / box_rows;
      // 64-dim blocks of this head in the map's rows (shared KV: V over the K rows)
      const int z0 = is_k ? it.kvh * H2 : it.kvh * ((P.kv_shared ? P.hk : HD) / 64);
      const int nslots = is_k ? kPfKSlots : kPfVSlots;
      uint64_t* fullb = is_k ? kfull : vfull;
      uint64_t* emptyb = is_k ? kempty : vempty;
      uint8_t* ring = is_k ? kring : vring;
      const CUtensorMap* map = is_k ? &tmk : &tmv;
      int iss = 0;
      bool ok = true;
      for (int n = 0; n < ntiles; ++n) {
        const int t0 = it.tok0 + n * kPfTok;
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
        const uint32_t bytes = uint32_t(npieces) * box_rows * 128 * H2;
        const int slot = iss % nslots;
        if (!mbar_wait(&emptyb[slot], ((iss / nslots) & 1) ^ 1)) {
          ok = false;
          break;
        }
        uint8_t* dst = ring + slot * Cfg::kSlot;
        uint64_t* full = &fullb[slot];
        if (bytes) mbar_arrive_expect_tx(full, bytes); else mbar_arrive(full);
        for (int pc = 0; pc < pieces; ++pc) {
          const int tok = t0 + pc * box_rows;
          if (tok >= it.tok1) break;
          const int ph = bt_row[tok / bs];
          if (ph < 0 || ph >= P.num_blocks) continue;
          const int row = ph * bs + tok % bs;
          if (box_rows == kPfTok) {
            // one box: [H2 halves][128 tokens][128 B] = the slot
            tma_load_3d(dst, map, full, 0, row, z0, pol);
          } else {
            for (int h = 0; h < H2; ++h)
              tma_load_3d(dst + h * kHalfK + pc * box_rows * 128, map, full, 0, row, z0 + h, pol);
          }
        }
        ++iss;
      }
      if (!ok) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
      for (int i = iss - nslots > 0 ? iss - nslots : 0; i < iss; ++i)
        mbar_wait(&fullb[i % nslots], (i / nslots) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer =================
    // Issues S(n) = Q . K(n)^T (into S buffer n & 1) and O += P(m) . V(m)
    // (into the O of tile m's group) in whatever order their inputs become
    // ready, so that one group's softmax never holds back the other's next
    // QK. Lane 0 polls; the warp follows its verdicts.
    bool ok = true;
    const uint32_t q_addr = smem_u32(q_s);
    const uint32_t k_addr = smem_u32(kring), v_addr = smem_u32(vring);
    if (ntiles > 0 && !warp_wait(q_ready, 0, lane)) ok = false;
    auto ready = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool r = lane == 0 ? mbar_try_wait(bar, parity) : false;
      return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
    };
    int nq = 0, np = 0;  // next QK tile, next PV tile
    long long idle_since = clock64();
    while (ok && np < ntiles) {
      bool progressed = false;
      // QK(nq): its K slot has landed, and its S buffer's P (tile nq - 2) was
      // read by PV(nq - 2): issued before this QK by this thread, which the
      // tensor cores carry out in order
      if (nq < ntiles && (nq < 2 || (np >= nq - 1 && ready(&s_free[nq & 1], ((nq >> 1) - 1) & 1))) &&
          ready(&kfull[nq % kPfKSlots], (nq / kPfKSlots) & 1)) {
        const int ks = nq % kPfKSlots;
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < H2; ++h) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t a = smem_desc(q_addr + h * kHalfQ + k * 32, 16, 1024);
              const uint64_t b = smem_desc(k_addr + ks * Cfg::kSlot + h * kHalfK + k * 32, 16, 1024);
              tc_mma(tmem_s + (nq & 1) * 128, a, b, kIdescQK, (h | k) != 0);
            }
          }
          tc_commit(&kempty[ks]);
          tc_commit(&s_full[nq & 1]);
        }
        __syncwarp();
        ++nq;
        progressed = true;
      }
      // PV(np): its P was written and its V slot has landed
      if (np < nq && ready(&p_full[np & 1], (np >> 1) & 1) &&
          ready(&vfull[np % kPfVSlots], (np / kPfVSlots) & 1)) {
        const int m = np, pb = m & 1, vs = m % kPfVSlots;
        const int nvalid = min(kPfTok, it.tok1 - (it.tok0 + m * kPfTok));
        if (nvalid < kPfTok) {
          // V rows past the range may hold anything (NaN included): zero them
          uint8_t* vb = vring + vs * Cfg::kSlot;
          const int per = (kPfTok - nvalid) * 8;  // 16-byte chunks per half
          for (int idx = lane; idx < H2 * per; idx += 32) {
            const int h = idx / per, rem = idx % per;
            *reinterpret_cast<uint4*>(vb + h * kHalfK + (nvalid + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < kPfTok / 16; ++k) {
            // A = P in TMEM: row m in lane m, 16 tokens = 8 columns of fp16 pairs
            // B = V (tokens x dims, MN-major: 64-dim halves kHalfK apart)
            const uint64_t b = smem_desc(v_addr + vs * Cfg::kSlot + k * 2048, kHalfK, 1024);
            tc_mma_tmem_a(tmem_o + pb * 128, tmem_s + pb * 128 + k * 8, b, kIdescPV, ((m >> 1) | k) != 0);
          }
          tc_commit(&vempty[vs]);
          tc_commit(&pv_done[pb]);
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
      tc_commit(qk_done);
      tc_commit(o_done);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ================= softmax: group g (warps 4-7 / 8-11) takes tiles n = g mod 2 =====
    // Each group keeps its own running max, sum and O accumulator (TMEM
    // columns 256 + 128 g); the two states of a row are merged at the end.
    const int grp = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const bool active = true;           // M=128: TMEM lane m holds row m
    const int r = quarter * 32 + lane;  // row of the tile
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const uint32_t o_mine = tmem_o + grp * 128 + lane_base;
    const bool row_ok = active && r < it.nrows;
    const int rr = it.r0 + r;
    const int qi = row_ok ? rr / G : 0;  // query token of the row
    const int p_row = prefix + qi;       // its position
    const float slope = (row_ok && P.mask_type == PA_MASK_ALIBI)
                            ? P.alibi_slopes[it.kvh * G + rr % G] * kLog2e : 0.f;
    if (grp == 0) {
      // Q tile: rows r, 64-dim halves, swizzled; 128 threads, 16-byte chunks
      const int st = tid - 128;
      constexpr int kChunks = kPfRows * (HD / 8);
      constexpr int kPer = kChunks / 128, kRound = kPer < 8 ? kPer : 8;
#pragma unroll
      for (int k0 = 0; k0 < kPer; k0 += kRound) {
        uint4 v[kRound];  // every load of the round before any store
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
          const int idx = st + (k0 + k) * 128;
          const int row = idx / (HD / 8), c = idx % (HD / 8);
          v[k] = make_uint4(0, 0, 0, 0);
          if (row < it.nrows) {
            const int rq = it.r0 + row;
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
      if (lane == 0) mbar_arrive(q_ready);
    }
    float m_ref = -INFINITY;  // reference max of the row over this group's tiles (base 2)
    float l = 0.f;            // sum of exp2(s - m_ref) over those keys
    bool ok = true;
    for (int n = grp; n < ntiles; n += 2) {
      const int b = n & 1;  // = grp: S, P and O buffers of this group
      if (!warp_wait(&s_full[b], (n >> 1) & 1, lane)) { ok = false; break; }
      tc_fence_after();
      // Pass 1, 32 columns at a time: scores in base 2 with the bias, written
      // back into the S buffer, and the tile's row max.
      const uint32_t sbuf = tmem_s + b * 128 + lane_base;
      const int j0 = it.tok0 + n * kPfTok;  // key of column 0
      const int jend = it.tok1 - j0;       // columns at or past this are outside the range
      float tmax = -INFINITY;
      // (tcgen05.ld / st are warp-collective: the branch below must be taken by
      // the whole warp, so the test is whether any row of the warp needs it)
      const bool diag_row = row_ok && j0 + kPfTok - 1 > p_row;
      if (P.mask_type == PA_MASK_NORM_COMPRESS && __any_sync(0xffffffffu, diag_row)) {
        // a tile reaching above some row's diagonal: read the mask there
        const int mr = min(max(p_row - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
        const __half* mrow = P.mask + mr * PA_COMPRESS_MASK_SIZE;
#pragma unroll 1
        for (int cc = 0; cc < kPfTok / 32; ++cc) {
          float x[32];
          tmem_ld32(sbuf + cc * 32, x);
          // the chunk's mask values, loaded together (indices clamped into the
          // mask, so every load is in bounds) and used only above the diagonal
          const bool need = __any_sync(0xffffffffu, diag_row && j0 + cc * 32 + 31 > p_row);
          __half mv[32];
          if (need) {
            const int m0 = j0 + cc * 32 - sigma;  // mask column of this chunk's first key
            if (m0 >= 0 && m0 + 32 <= PA_COMPRESS_MASK_SIZE && (m0 & 7) == 0) {
              // 64 contiguous bytes of the row, 16-byte aligned: four vector loads
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
        // no bias (or a tile wholly on or below the diagonal)
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
      if (n >= 2 && !__all_sync(0xffffffffu, mbar_wait(&pv_done[b], ((n - 2) >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Pass 2: probabilities as fp16 pairs into the S buffer's first 64
      // columns, where the PV MMA reads them: chunk cc's 32 scores (columns
      // 32cc..) become columns 16cc.., all of which this thread has read.
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
      if (lane == 0) mbar_arrive(&s_free[b]);
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
      if (lane == 0) mbar_arrive(&p_full[b]);
    }
    if (!ok && lane == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    launch_dependents();
    // ---- merge the two groups' states per row, then O / l
    float* xm = reinterpret_cast<float*>(smem + Cfg::xchg_off);  // [2][rows]: group 1's m and l
    if (grp == 1 && active) {
      xm[r] = m_ref;
      xm[kPfRows + r] = l;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");  // the 8 softmax warps
    if (grp == 0) {
      const bool got = ok && warp_wait(o_done, 0, lane);
      const bool partial = it.slot >= 0;
      const bool fits = !partial || int64_t(it.slot) + it.nrows <= P.part_rows_cap;
      if (!fits && r == 0) set_status(P.status, PA_STATUS_BIT_WORKSPACE);
      if (got && fits) {
        tc_fence_after();
        const bool two = ntiles >= 2;  // group 1 ran (and wrote its O)
        const float m1 = two ? xm[r] : -INFINITY, l1 = two ? xm[kPfRows + r] : 0.f;
        const float mm = fmaxf(m_ref, m1);
        const float a0 = ntiles > 0 ? ex2(m_ref - mm) : 0.f, a1 = two ? ex2(m1 - mm) : 0.f;
        const float lt = l * a0 + l1 * a1;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const float w0 = a0 * inv, w1 = a1 * inv;
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          float o[32], o1[32];
          tmem_ld32(tmem_o + c * 32 + lane_base, o);
          if (two) tmem_ld32(tmem_o + 128 + c * 32 + lane_base, o1);
          tmem_wait_ld();
          if (!row_ok) continue;
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = (ntiles > 0 ? o[i] * w0 : 0.f) + (two ? o1[i] * w1 : 0.f);
          if (partial) {
            uint4* dst = reinterpret_cast<uint4*>(P.part_o + (int64_t(it.slot) + r) * HD + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 pk;
              pk.x = pack_half2(o[8 * i + 0], o[8 * i + 1]);
              pk.y = pack_half2(o[8 * i + 2], o[8 * i + 3]);
              pk.z = pack_half2(o[8 * i + 4], o[8 * i + 5]);
              pk.w = pack_half2(o[8 * i + 6], o[8 * i + 7]);
              dst[i] = pk;
            }
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
        if (partial && row_ok) P.part_lse[it.slot + r] = lt > 0.f ? (mm + log2f(lt)) * kLn2 : -INFINITY;
      }
    }
  }
  // ---- teardown: every tcgen05 op has completed before TMEM is freed
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      mbar_wait(qk_done, 0);
      mbar_wait(o_done, 0);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols));
  }
}

cudaError_t launch_pf(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                      int64_t n_items, cudaStream_t stream);

}  // namespace pa
