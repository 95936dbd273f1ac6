// Paged attention for 256-row tiles (prefill, q = L, and any launch whose
// group rows G * max_q exceed 128) on the tcgen05 tensor cores: two 128-row
// query tiles per CTA share every K and V tile. Same operation, work item and
// split/merge contract as the other kernels (PagedAttentionOperation
// semantics; task list and FlashDecode merge of the SparseAttnSharedkvMetadata
// page).
//
// One CTA per work item, 128-token key tiles, 12 warps:
//   warps 0, 2 TMA producers of K and of V (3-D boxes, 128-byte swizzle) into
//              a 3-slot K ring and a 2- or 3-slot V ring; a slot is released
//              by the last MMA that reads it (a key tile past one query
//              tile's causal range has one reader).
//   warp 1     allocates TMEM; one thread issues, for each query tile g,
//              S_g = Q_g . K^T (M=128 rows, N=128 tokens, K-major operands)
//              and O_g += P_g . V (A = P_g from TMEM, B = V MN-major) in a
//              fixed order with blocking waits. S_g(n + 1) overwrites the
//              columns that held P_g(n), so it is issued after PV_g(n); the
//              other tile's chain fills the tensor pipe meanwhile.
//   warps 4-11 softmax group g (warps 4-7: g = 0, 8-11: g = 1) owns query tile
//              g over every key tile: one row per thread (TMEM lane m holds
//              row m of an M=128 accumulator), scores from TMEM in 32-column
//              loads, the reference max moved (and O_g rescaled in TMEM) only
//              when a score passes it by more than 2^8, P_g written as fp16
//              pairs into the S_g columns.
//   warp 3     no role.
// TMEM: S_g at columns [128 g, 128 g + 128), O_g at [256 + 128 g, ...).
// With the compressed causal mask each query tile stops after its last row's
// position, and only keys above the diagonal read the mask. Every wait is
// bounded; on a timeout the CTA records PA_STATUS_BIT_TIMEOUT and exits
// cleanly.
#pragma once

#include "pa_prefill_tc.cuh"

namespace pa {

constexpr int kPpRows = PA_PF_PAIR_ROWS;  // rows of a work item (two query tiles)
constexpr int kPpQRows = kPpRows / 2;     // rows of one query tile (M of the MMAs)
constexpr int kPpThreads = 384;

template <int HD>
struct PpCfg {
  static constexpr int kHalves = HD / 64;
  static constexpr int kKSlots = 3;
  static constexpr int kVSlots = HD == 128 ? 2 : 3;  // what the shared memory leaves
  static constexpr uint32_t kSlot = uint32_t(kPfTok) * HD * 2;  // one K or V tile
  static constexpr uint32_t kQt = uint32_t(kPpQRows) * HD * 2;  // one query tile
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t k_off = q_off + 2 * kQt;
  static constexpr uint32_t v_off = k_off + kKSlots * kSlot;
  static constexpr uint32_t bars_off = v_off + kVSlots * kSlot;
  static constexpr int kBars = 2 * (kKSlots + kVSlots) + 12;
  static constexpr uint32_t tmem_slot_off = bars_off + kBars * 8;
  static constexpr uint32_t bytes = tmem_slot_off + 16 + 1024;
  static_assert(bytes <= kTcMaxSmem, "shared memory");
  static_assert(k_off % 1024 == 0 && v_off % 1024 == 0, "128-byte swizzle atoms");
};

template <int HD>
__global__ void __launch_bounds__(kPpThreads, 1) pf_pair_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
    const FwdParams P) {
  using Cfg = PpCfg<HD>;
  constexpr int H2 = Cfg::kHalves;
  constexpr int kK = Cfg::kKSlots, kV = Cfg::kVSlots;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdescQK = mma_idesc(kPpQRows, kPfTok, 0, 0);
  constexpr uint32_t kIdescPV = mma_idesc(kPpQRows, HD, 0, 1);
  constexpr uint32_t kHalfK = uint32_t(kPfTok) * 128;    // one 64-dim half of a K/V tile
  constexpr uint32_t kHalfQ = uint32_t(kPpQRows) * 128;  // one 64-dim half of a query tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* q_s = smem + Cfg::q_off;
  uint8_t* kring = smem + Cfg::k_off;
  uint8_t* vring = smem + Cfg::v_off;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + Cfg::bars_off);
  uint64_t* kempty = kfull + kK;
  uint64_t* vfull = kempty + kK;
  uint64_t* vempty = vfull + kV;
  uint64_t* s_full = vempty + kV;  // [2] S_g written
  uint64_t* p_full = s_full + 2;   // [2] P_g written (and O_g rescaled)
  uint64_t* pv_done = s_full + 4;  // [2] PV_g complete
  uint64_t* qk_done = s_full + 6;
  uint64_t* o_done = s_full + 7;
  uint64_t* q_ready = s_full + 8;  // both query tiles in shared memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::tmem_slot_off);

  if (P.counts && int(blockIdx.x) >= P.counts[0]) return;  // past a device plan's items
  // Items run last to first: the later row tiles of a causal sequence meet
  // more keys, so the longest items start first.
  const int n_items = P.counts ? P.counts[0] : int(gridDim.x);
  Item it;
  it.load(P, n_items - 1 - int(blockIdx.x));
  const int G = P.group, bs = P.block_size;
  const int prefix = it.L - it.qlen;
  // key tiles of each query tile: all of the item's range, or with the
  // compressed causal mask up to the tile's last row's position (later keys
  // carry the mask's fill for every row of that tile)
  int nt[2];
  int tok1 = it.tok0;
  for (int g = 0; g < 2; ++g) {
    const int rows = min(kPpQRows, it.nrows - g * kPpQRows);
    int t1 = it.tok0;
    if (rows > 0) {
      t1 = it.tok1;
      if (P.mask_type == PA_MASK_NORM_COMPRESS) {
        const int pmax = prefix + (it.r0 + g * kPpQRows + rows - 1) / G;
        t1 = max(it.tok0, min(it.tok1, pmax + 1));
      }
    }
    nt[g] = t1 > it.tok0 ? (t1 - it.tok0 + kPfTok - 1) / kPfTok : 0;
    tok1 = max(tok1, t1);
  }
  it.tok1 = tok1;
  const int ntiles = max(nt[0], nt[1]);
  const int sigma = it.L > PA_COMPRESS_MASK_SIZE ? it.L - PA_COMPRESS_MASK_SIZE : 0;

  if (tid == 0) {
    for (int s = 0; s < kK; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < kV; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&s_full[g], 1);
      mbar_init(&p_full[g], 4);
      mbar_init(&pv_done[g], 1);
    }
    mbar_init(qk_done, 1);
    mbar_init(o_done, 1);
    mbar_init(q_ready, 8);
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
  const uint32_t tmem_s = tmem;        // S_g: columns [128 g, 128 g + 128)
  const uint32_t tmem_o = tmem + 256;  // O_g: columns [256 + 128 g, 256 + 128 g + HD)

  if (warp == 0 || warp == 2) {
    // ================= TMA producers (lane 0): K (warp 0), V (warp 2) =========
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
      const int nslots = is_k ? kK : kV;
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
            tma_load_3d(dst, map, full, 0, row, z0, pol);  // [H2 halves][128 tokens][128 B]
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
    // A fixed order with blocking waits (no polling, which would take issue
    // slots from the softmax warps of this scheduler):
    //   S_0(0) S_1(0), then per key tile n:
    //   O_0 += P_0(n) V(n), S_0(n + 1), O_1 += P_1(n) V(n), S_1(n + 1)
    // S_g(n + 1) overwrites the columns that held P_g(n), so it follows
    // PV_g(n); the tensor pipe runs one thread's MMAs in order. A key tile
    // past one query tile's causal range is skipped for that tile; a K or V
    // slot is released after its last reader.
    bool ok = true;
    const uint32_t q_addr = smem_u32(q_s);
    const uint32_t k_addr = smem_u32(kring), v_addr = smem_u32(vring);
    if (ntiles > 0 && !warp_wait(q_ready, 0, lane)) ok = false;
    auto qk = [&](int g, int n) {
      const int ks = n % kK;
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < H2; ++h) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t a = smem_desc(q_addr + g * Cfg::kQt + h * kHalfQ + k * 32, 16, 1024);
            const uint64_t b = smem_desc(k_addr + ks * Cfg::kSlot + h * kHalfK + k * 32, 16, 1024);
            tc_mma(tmem_s + g * 128, a, b, kIdescQK, (h | k) != 0);
          }
        }
        tc_commit(&s_full[g]);
        // last reader of K(n): query tile 1 if it needs the tile, else tile 0
        if (g == 1 || n >= nt[1]) tc_commit(&kempty[ks]);
      }
      __syncwarp();
    };
    auto pv = [&](int g, int m) {
      const int vs = m % kV;
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kPfTok / 16; ++k) {
          // A = P_g in TMEM (16 tokens = 8 columns of fp16 pairs), B = V
          const uint64_t b = smem_desc(v_addr + vs * Cfg::kSlot + k * 2048, kHalfK, 1024);
          tc_mma_tmem_a(tmem_o + g * 128, tmem_s + g * 128 + k * 8, b, kIdescPV, (m | k) != 0);
        }
        tc_commit(&pv_done[g]);
        if (g == 1 || m >= nt[1]) tc_commit(&vempty[vs]);
      }
      __syncwarp();
    };
    // K(n) landed (waited once per tile, before its first QK)
    auto k_ready = [&](int n) { return warp_wait(&kfull[n % kK], (n / kK) & 1, lane); };
    if (ok && ntiles > 0) {
      if (!k_ready(0)) ok = false;
      tc_fence_after();
      for (int g = 0; g < 2 && ok; ++g)
        if (nt[g] > 0) qk(g, 0);
    }
    for (int n = 0; n < ntiles && ok; ++n) {
      // V(n) landed; rows past the range may hold anything (NaN included):
      // zero them before the first PV reads the tile
      if (!warp_wait(&vfull[n % kV], (n / kV) & 1, lane)) { ok = false; break; }
      const int nvalid = min(kPfTok, it.tok1 - (it.tok0 + n * kPfTok));
      if (nvalid < kPfTok) {
        uint8_t* vb = vring + (n % kV) * Cfg::kSlot;
        const int per = (kPfTok - nvalid) * 8;  // 16-byte chunks per half
        for (int idx = lane; idx < H2 * per; idx += 32) {
          const int h = idx / per, rem = idx % per;
          *reinterpret_cast<uint4*>(vb + h * kHalfK + (nvalid + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
        __syncwarp();
      }
      const bool next_k = n + 1 < ntiles;
      bool k_waited = false;
      for (int g = 0; g < 2; ++g) {
        if (n >= nt[g]) continue;
        if (!warp_wait(&p_full[g], n & 1, lane)) { ok = false; break; }
        tc_fence_after();
        pv(g, n);
        if (n + 1 < nt[g]) {
          if (next_k && !k_waited) {
            if (!k_ready(n + 1)) { ok = false; break; }
            k_waited = true;
            tc_fence_after();
          }
          qk(g, n + 1);
        }
      }
    }
    if (!ok && lane == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    if (lane == 0) {
      tc_commit(qk_done);
      tc_commit(o_done);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ================= softmax: group g (warps 4-7 / 8-11) owns query tile g =====
    const int grp = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int tr = quarter * 32 + lane;  // row of query tile grp = TMEM lane
    const int r = grp * kPpQRows + tr;   // row of the item
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const uint32_t o_mine = tmem_o + grp * 128 + lane_base;
    const bool row_ok = r < it.nrows;
    const int rr = it.r0 + r;
    const int qi = row_ok ? rr / G : 0;  // query token of the row
    const int p_row = prefix + qi;       // its position
    const float slope = (row_ok && P.mask_type == PA_MASK_ALIBI)
                            ? P.alibi_slopes[it.kvh * G + rr % G] * kLog2e : 0.f;
    {
      // query tile grp: rows, 64-dim halves, swizzled; 128 threads, 16-byte chunks
      const int st = tid - 128 - grp * 128;
      uint8_t* qt = q_s + grp * Cfg::kQt;
      constexpr int kChunks = kPpQRows * (HD / 8);
      constexpr int kPer = kChunks / 128, kRound = kPer;  // every load in flight at once
#pragma unroll
      for (int k0 = 0; k0 < kPer; k0 += kRound) {
        uint4 v[kRound];  // every load of the round before any store
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
          const int idx = st + (k0 + k) * 128;
          const int row = idx / (HD / 8), c = idx % (HD / 8);
          v[k] = make_uint4(0, 0, 0, 0);
          if (grp * kPpQRows + row < it.nrows) {
            const int rq = it.r0 + grp * kPpQRows + row;
            v[k] = *reinterpret_cast<const uint4*>(
                P.query + (int64_t(it.q_start + rq / G) * P.num_heads + it.kvh * G + rq % G) * HD + c * 8);
          }
        }
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
          const int idx = st + (k0 + k) * 128;
          const int row = idx / (HD / 8), c = idx % (HD / 8);
          *reinterpret_cast<uint4*>(qt + (c >> 3) * kHalfQ + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = v[k];
        }
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
    }
    float m_ref = -INFINITY;  // reference max of the row (base 2)
    float l = 0.f;            // sum of exp2(s - m_ref) over the row's keys so far
    bool ok = true;
    const uint32_t sbuf = tmem_s + grp * 128 + lane_base;
    const int my_tiles = grp ? nt[1] : nt[0];
    for (int n = 0; n < my_tiles; ++n) {
      if (!warp_wait(&s_full[grp], n & 1, lane)) { ok = false; break; }
      tc_fence_after();
      const int j0 = it.tok0 + n * kPfTok;  // key of column 0
      const int jend = it.tok1 - j0;       // columns at or past this are outside the range
      // (tcgen05.ld / st are warp-collective: the branches below must be taken
      // by the whole warp, so the test is whether any row of the warp needs
      // the mask)
      const bool diag_row = row_ok && j0 + kPfTok - 1 > p_row;
      const bool diag = P.mask_type == PA_MASK_NORM_COMPRESS && __any_sync(0xffffffffu, diag_row);
      // move the reference only when a score passes it by more than 2^8, and
      // order this thread's TMEM accesses after PV_g(n - 1), which read
      // P_g(n - 1) and wrote O_g (S_g(n) was issued after it, so it is done)
      bool grow = false;
      float alpha = 1.f;
      auto settle = [&](float tmax) -> bool {
        grow = tmax > m_ref + kTcRescaleThreshold;
        if (grow) {
          alpha = ex2(m_ref - tmax);  // 0 on the first tile
          m_ref = tmax;
          l *= alpha;
        }
        if (n >= 1 && !__all_sync(0xffffffffu, mbar_wait(&pv_done[grp], (n - 1) & 1))) return false;
        tc_fence_after();
        return true;
      };
      if (!diag && P.mask_type != PA_MASK_ALIBI && P.mask_type != PA_MASK_NORM) {
        // No bias on this tile: one pass. The 128 scores come from TMEM with
        // every load in flight at once; the row max is taken on the raw
        // products (rounding is monotonic and the scale positive, so it
        // equals the max of the scaled scores); P = exp2(x * scale - m) is
        // written as fp16 pairs into the first 64 columns of S_g.
        float x[kPfTok];
#pragma unroll
        for (int cc = 0; cc < kPfTok / 32; ++cc) tmem_ld32(sbuf + cc * 32, x + cc * 32);
        tmem_wait_ld();
        if (jend < kPfTok) {
#pragma unroll
          for (int i = 0; i < kPfTok; ++i) x[i] = i < jend ? x[i] : -INFINITY;
        }
        float t4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four max chains
#pragma unroll
        for (int i = 0; i < kPfTok; ++i) t4[i & 3] = fmaxf(t4[i & 3], x[i]);
        const float tmax = fmaxf(fmaxf(t4[0], t4[1]), fmaxf(t4[2], t4[3])) * P.scale_log2;
        if (!settle(tmax)) { ok = false; break; }
        // exponents and sums on packed fp32 pairs (two lanes per instruction)
        const float2 sc2 = make_float2(P.scale_log2, P.scale_log2);
        const float2 nm2 = make_float2(-m_ref, -m_ref), one2 = make_float2(1.f, 1.f);
        float2 ps2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // four sum chains
#pragma unroll
        for (int cc = 0; cc < kPfTok / 32; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 a = fma2(make_float2(x[cc * 32 + 2 * i], x[cc * 32 + 2 * i + 1]), sc2, nm2);
            const float e0 = ex2(a.x), e1 = ex2(a.y);
            ps2[i & 1] = fma2(make_float2(e0, e1), one2, ps2[i & 1]);
            pk[i] = pack_half2(e0, e1);
          }
          tmem_st16u(sbuf + cc * 16, pk);
        }
        l += (ps2[0].x + ps2[0].y) + (ps2[1].x + ps2[1].y);
        tmem_wait_st();
      } else {
        // Pass 1, 32 columns at a time: scores in base 2 with the bias,
        // written back into S_g, and the tile's row max.
        float tmax = -INFINITY;
        if (diag) {
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
        } else {
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
        }
        tmem_wait_st();
        if (!settle(tmax)) { ok = false; break; }
        // Pass 2: probabilities as fp16 pairs into the first 64 columns of S_g,
        // where the PV MMA reads them: chunk cc's 32 scores (columns 32cc..)
        // become columns 16cc.., all of which this thread has read.
        float ps[4] = {0.f, 0.f, 0.f, 0.f};  // four independent sum chains
#pragma unroll 1
        for (int cc = 0; cc < kPfTok / 32; ++cc) {
          float x[32];
          tmem_ld32(sbuf + cc * 32, x);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float e0 = ex2(x[2 * i] - m_ref), e1 = ex2(x[2 * i + 1] - m_ref);
            ps[(2 * i) & 3] += e0;
            ps[(2 * i + 1) & 3] += e1;
            pk[i] = pack_half2(e0, e1);
          }
          tmem_st16u(sbuf + cc * 16, pk);
        }
        l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        tmem_wait_st();
      }
      if (n >= 1 && __any_sync(0xffffffffu, grow && row_ok)) {
        // rescale this warp's rows of O_g (rows that did not grow use 1)
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
      if (lane == 0) mbar_arrive(&p_full[grp]);
    }
    if (!ok && lane == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    launch_dependents();
    // ---- epilogue: O_g / l for this group's rows
    const bool got = ok && warp_wait(o_done, 0, lane);
    const bool partial = it.slot >= 0;
    const bool fits = !partial || int64_t(it.slot) + it.nrows <= P.part_rows_cap;
    if (!fits && r == 0) set_status(P.status, PA_STATUS_BIT_WORKSPACE);
    if (got && fits) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool any = my_tiles > 0;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        tmem_ld32(o_mine + c * 32, o);
        tmem_wait_ld();
        if (!row_ok) continue;
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = any ? o[i] * inv : 0.f;
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
      if (partial && row_ok) P.part_lse[it.slot + r] = (any && l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
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

cudaError_t launch_pf_pair(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                           int64_t n_items, cudaStream_t stream);

}  // namespace pa
