// Split-KV paged decode for 16-row tiles over a shared-KV cache whose V is
// the first hv dims of each K row (the latent cache of 576-dim rows over a
// 512-dim V, or hk = hv = 256 / 512), on the warp-level MMA.
// PagedAttentionOperation incremental phase (576/512 heads) with the shared
// K/V alias of SparseAttnSharedkvMetadata's parameter table; the split/merge
// structure follows SparseAttnSharedkvMetadata.
//
// Why not tcgen05 for this shape: with 16 rows the QK^T of a 64-token tile is
// 36 MMAs of N = 16 at hk = 576 and the PV 16 more, and a tcgen05.mma of that
// size costs about 50 cycles (a floor measured for M <= 128, N <= 64); the
// slots of the shared cache stay held through QK -> softmax -> PV, and that
// chain cannot overlap enough. mma.sync m16n8k16 ran at 2 cycles per
// instruction per SM (21 cycles of latency, ldmatrix 39), so the same tile is
// 544 of them, ~1100 cycles.
//
// One CTA per SM: a TMA producer warp and 8 compute warps over a ring of
// whole-tile slots, [hk/64 halves][64 tokens][128 B] with the 128-byte
// swizzle, each filled by one TMA box per tile (per block piece below
// 64-token blocks): few, large copies, since each copy costs the issuing
// thread time on a busy SM (measured: 8 KB boxes stream at 70 GB/s per SM
// beside 16 busy warps, 16-32 KB boxes at 127-142 GB/s). Three 73.7 KB slots
// for 576-dim rows let a tile's copy start two tiles ahead. Nine warps leave
// each thread 168 registers: a compute warp keeps the query fragments of both
// 8-row halves of its dims, so every K element is read from shared memory
// once. Per tile:
//   A. QK: warp (tq, dh) = (w & 3, w >> 2) forms the partial S^T of tokens
//      16 tq.., all 16 rows, dims dh * hk/2.. (A = K via ldmatrix, one
//      operand for the two 8-row MMAs, B = its Q^T fragments, in registers
//      for the whole item) into shared memory.
//   B. softmax: warp w owns rows w and w + 8: the two partials of its 64
//      scores summed, scaled, biased and masked, the running max, p = 2^(s - m)
//      in fp16 into P[16][64] and the row's rescale factor. P lives in the
//      tile's dims past hv (read only by QK) when there are any.
//   C. PV: warp w owns dims w * hv/8..: O^T *= alpha, O^T += V^T P^T (V^T via
//      ldmatrix.trans, P^T via ldmatrix); O^T in registers for the whole item.
// Two named barriers (the 8 compute warps) separate the phases; a slot returns
// to the producer when every compute warp is past its PV.
#pragma once

#include "pa_decode_mma.cuh"

namespace pa {

constexpr int kWideWarps = 8;                        // compute warps
constexpr int kWideThreads = (kWideWarps + 1) * 32;  // + the producer warp
constexpr int kWideTok = 64;                         // tokens per tile
constexpr uint32_t kWideHalfBytes = kWideTok * 128;  // 64 tokens x 64 dims
constexpr int kWidePsStride = 68;  // floats per row of a partial S^T (64 + 4: no bank conflicts)
constexpr uint32_t kWideMaxSmem = 232448;

// Shared-KV head-size pairs of the kernel.
inline bool wide_supported(int hk, int hv, bool shared_kv) {
  return shared_kv && ((hk == 576 && hv == 512) || (hk == hv && (hk == 256 || hk == 512)));
}

template <int HK, int HV>
struct WideCfg {
  static constexpr int kHalves = HK / 64;
  static constexpr uint32_t kTileBytes = kHalves * kWideHalfBytes;
  static constexpr bool kPInTile = HK - HV >= 64;  // P in the tile's QK-only dims
  static constexpr uint32_t kPsBytes = 2 * 16 * kWidePsStride * 4;  // [dh][row][token] fp32
  static constexpr uint32_t kPBytes = kPInTile ? 0 : 16 * 128;      // P [row][64 tokens] fp16
  static constexpr uint32_t kRowBytes = 3 * 16 * 4;                  // alpha, l, m per row
  static constexpr uint32_t kFixed = kPsBytes + kPBytes + kRowBytes + 2 * 8 * 8;
  static constexpr int kFit = int((kWideMaxSmem - 1024 - kFixed) / kTileBytes);
  static constexpr int kSlots = kFit < 6 ? kFit : 6;
  static constexpr uint32_t ring_off = 0;  // 1024-aligned (128-byte swizzle atoms)
  static constexpr uint32_t ps_off = ring_off + kSlots * kTileBytes;
  static constexpr uint32_t p_off = ps_off + kPsBytes;  // unused when kPInTile
  static constexpr uint32_t rows_off = p_off + kPBytes;
  static constexpr uint32_t bars_off = rows_off + kRowBytes;  // full[kSlots], empty[kSlots]
  static constexpr uint32_t bytes = bars_off + 16 * kSlots + 1024;  // + alignment slack
  static_assert(kSlots >= 2, "two tiles must fit");
  static_assert(bytes <= kWideMaxSmem, "shared memory");
};

// Named barrier 1 over the compute warps, returning the OR of `pred`: all of
// them take the same continue/abort decision.
__device__ __forceinline__ bool wide_bar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(uint32_t(pred))
      : "memory");
  return r != 0;
}

// tmk: the cache as a 3-D map (64 dims, token rows, 64-dim blocks) whose box
// is 64 tokens x hk/64 blocks when the block size is a multiple of 64, else
// box_rows tokens x one block.
template <int HK, int HV>
__global__ void __launch_bounds__(kWideThreads, 1) wide_decode_kernel(
    const __grid_constant__ CUtensorMap tmk, const FwdParams P) {
  using Cfg = WideCfg<HK, HV>;
  constexpr int NH = Cfg::kHalves, VH = HV / 64;
  constexpr int KSH = HK / 32;   // 16-dim k-steps of one dim half
  constexpr int MTW = HV / 128;  // 16-dim m-tiles of one warp's PV slice
  constexpr int NT = Cfg::kSlots;
  constexpr int NTH = kWideWarps * 32;  // compute threads
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* ring = smem + Cfg::ring_off;
  float* ps = reinterpret_cast<float*>(smem + Cfg::ps_off);
  float* alpha_s = reinterpret_cast<float*>(smem + Cfg::rows_off);
  float* l_s = alpha_s + 16;
  float* m_s = l_s + 16;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::bars_off);
  uint64_t* empty = full + NT;

  if (P.counts && int(blockIdx.x) >= P.counts[0]) return;  // past a device plan's items
  Item it;
  it.load(P, blockIdx.x);
  const int G = P.group, bs = P.block_size;
  const int prefix = it.L - it.qlen;
  if (P.mask_type == PA_MASK_NORM_COMPRESS && it.nrows > 0) {
    // Causal trim: keys past the last row's position have probability exactly
    // zero in fp32 (a large negative fill); the item stops before them.
    const int pmax = prefix + (it.r0 + it.nrows - 1) / G;
    it.tok1 = max(it.tok0, min(it.tok1, pmax + 1));
  }
  const int ntok = it.tok1 - it.tok0;
  const int ntiles = ntok > 0 ? (ntok + kWideTok - 1) / kWideTok : 0;

  if (tid == 0) {
    for (int s = 0; s < NT; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWideWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWideWarps) {
    // ================= TMA producer =================
    // Lane 0 waits for free slots and issues the copies; the warp keeps the
    // item's block-table entries in registers, 32 blocks a batch and one
    // batch ahead, so that no copy waits for a dependent global load.
    if (ntiles > 0) {
      const int32_t* bt_row = P.block_tables + int64_t(it.b) * P.max_blocks_per_seq;
      // the largest power of two dividing both the block and the tile
      const int box_rows = (bs & -bs) < kWideTok ? (bs & -bs) : kWideTok;
      const int pieces = kWideTok / box_rows;  // <= 4 (block sizes are multiples of 16)
      const int nblk = (it.tok1 - 1) / bs - it.kb0 + 1;  // blocks the item reads
      auto fetch = [&](int batch) {
        const int rb = 32 * batch + lane;
        return rb < nblk ? __ldg(bt_row + it.kb0 + rb) : -1;
      };
      int batch = 0, cur = fetch(0), nxt = fetch(1);
      const int z0 = it.kvh * NH;
      const uint64_t pol = policy_evict_first();
      bool ok = true;
      int issued = 0;
      for (int n = 0; n < ntiles && ok; ++n) {
        const int t0 = it.tok0 + n * kWideTok;
        int rws[4];
        int npieces = 0;
        for (int pc = 0; pc < pieces; ++pc) {
          const int tok = t0 + pc * box_rows;
          rws[pc] = -1;
          if (tok >= it.tok1) continue;  // warp-uniform
          const int rb = tok / bs - it.kb0;
          while ((rb >> 5) > batch) {
            cur = nxt;
            nxt = fetch(batch + 2);
            ++batch;
          }
          const int ph = __shfl_sync(0xffffffffu, cur, rb & 31);
          if (ph < 0 || ph >= P.num_blocks) {
            if (lane == 0) set_status(P.status, PA_STATUS_BIT_BLOCK_INDEX);
            continue;
          }
          rws[pc] = ph * bs + tok % bs;
          ++npieces;
        }
        if (lane == 0) {
          const int slot = n % NT;
          ok = mbar_wait(&empty[slot], ((n / NT) & 1) ^ 1, P.wait_limit);
          if (ok) {
            const uint32_t bytes = uint32_t(npieces) * box_rows * 128 * NH;
            if (bytes) {
              mbar_arrive_expect_tx(&full[slot], bytes);
            } else {
              mbar_arrive(&full[slot]);
            }
            uint8_t* dst = ring + slot * Cfg::kTileBytes;
            for (int pc = 0; pc < pieces; ++pc) {
              if (rws[pc] < 0) continue;
              if (box_rows == kWideTok) {
                // one box: [NH halves][64 tokens][128 B] = the slot
                tma_load_3d(dst, &tmk, &full[slot], 0, rws[pc], z0, pol);
              } else {
                for (int h = 0; h < NH; ++h)
                  tma_load_3d(dst + h * kWideHalfBytes + pc * box_rows * 128, &tmk, &full[slot], 0,
                              rws[pc], z0 + h, pol);
              }
            }
            ++issued;
          }
          // tiles 0 and 1 first: at the start of a wave every CTA's ring is
          // empty, and the first tile would otherwise queue behind the third
          // of every CTA (tile 2 is issued once tile 0 has landed)
          if (ok && n == 1 && ntiles > 2) ok = mbar_wait(&full[0], 0, P.wait_limit);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
      if (lane == 0) {
        if (!ok) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
        // let every issued copy land before the CTA can exit (default limit)
        for (int i = issued - NT > 0 ? issued - NT : 0; i < issued; ++i)
          mbar_wait(&full[i % NT], (i / NT) & 1);
      }
    }
    return;
  }

  // ================= compute warps =================
  const int g = lane >> 2, c = lane & 3;
  const int tq = warp & 3, dh = warp >> 2;
  const int li = lane >> 3, lr = lane & 7;  // ldmatrix: matrix and row this lane addresses

  // Q^T fragments of this warp's dim half: B[k = dim][n = row], rows 8 j + g.
  uint32_t qf[KSH][2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int row = j * 8 + g;
    const bool rok = row < it.nrows;
    const int rr = it.r0 + row;
    const __half* qrow =
        P.query + (int64_t(it.q_start + (rok ? rr / G : 0)) * P.num_heads + it.kvh * G + (rok ? rr % G : 0)) * HK;
#pragma unroll
    for (int ks = 0; ks < KSH; ++ks) {
      const int d0 = (dh * KSH + ks) * 16;
      qf[ks][j][0] = rok ? *reinterpret_cast<const uint32_t*>(qrow + d0 + 2 * c) : 0u;
      qf[ks][j][1] = rok ? *reinterpret_cast<const uint32_t*>(qrow + d0 + 8 + 2 * c) : 0u;
    }
  }
  // Rows of phase B (warp w: rows w and w + 8) and their constants.
  int prow[2];
  float slope2[2], m_run[2], l_lane[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = warp + 8 * h;
    const bool rok = r < it.nrows;
    prow[h] = rok ? prefix + (it.r0 + r) / G : it.L - 1;
    slope2[h] = (rok && P.mask_type == PA_MASK_ALIBI)
                    ? P.alibi_slopes[it.kvh * G + (it.r0 + r) % G] * kLog2e
                    : 0.f;
    m_run[h] = -INFINITY;
    l_lane[h] = 0.f;
  }
  const int sigma = it.L > PA_COMPRESS_MASK_SIZE ? it.L - PA_COMPRESS_MASK_SIZE : 0;
  // Per-lane parts of the ldmatrix addresses. QK: token row 16 tq + 8 (li & 1)
  // + lr; the 16-byte chunk of k-step K is (2 (K & 3) + (li >> 1)) ^ lr, whose
  // terms sit on disjoint bits. PV: token row 8 (li >> 1) + lr of a 16-token
  // step, chunk (vch + 2 mt + (li & 1)) ^ lr, again on disjoint bits.
  const uint32_t a_row = uint32_t(tq * 16 + (li & 1) * 8 + lr) * 128;
  const uint32_t a_chk = uint32_t((li >> 1) ^ lr);
  const int vd0 = warp * (HV / kWideWarps);
  const int vh = vd0 >> 6, vch = (vd0 & 63) >> 3;
  const uint32_t v_row = uint32_t((li >> 1) * 8 + lr) * 128;
  const uint32_t v_chk = uint32_t((vch + (li & 1)) ^ lr);
  const uint32_t p_row = v_row;  // P row this lane addresses: the same pattern
  const uint32_t p_chk = uint32_t((li & 1) ^ lr);
  float o[MTW][2][4];
#pragma unroll
  for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
    for (int j = 0; j < 2; ++j) o[mt][j][0] = o[mt][j][1] = o[mt][j][2] = o[mt][j][3] = 0.f;

  bool ok = true;
  for (int n = 0; n < ntiles; ++n) {
    const int slot = n % NT;
    uint8_t* tile = ring + slot * Cfg::kTileBytes;
    // P of this tile: its QK-only dims, else the separate buffer
    uint8_t* p_s = Cfg::kPInTile ? tile + VH * kWideHalfBytes : smem + Cfg::p_off;
    // ---- A: partial S^T of tokens 16 tq.., rows 0-15, this warp's dim half
    if (ok && !__all_sync(0xffffffffu, mbar_wait_own(&full[slot], (n / NT) & 1, P.wait_limit)))
      ok = false;
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (ok) {
      // one K operand feeds both 8-row MMAs (two accumulator chains); each
      // operand is loaded two k-steps ahead of its MMAs
      const uint8_t* ab = tile + a_row;
      auto a_addr = [&](int ks) {
        const int K = dh * KSH + ks;
        return ab + (K >> 2) * kWideHalfBytes + ((a_chk ^ uint32_t((K & 3) << 1)) << 4);
      };
      uint32_t a[2][4];
      ldsm_x4(a[0], a_addr(0));
      ldsm_x4(a[1], a_addr(1));
#pragma unroll
      for (int ks = 0; ks < KSH; ++ks) {
        mma_16816(s[0], a[ks & 1], qf[ks][0][0], qf[ks][0][1]);
        mma_16816(s[1], a[ks & 1], qf[ks][1][0], qf[ks][1][1]);
        if (ks + 2 < KSH) ldsm_x4(a[ks & 1], a_addr(ks + 2));
      }
    }
    {
      float* pq = ps + dh * 16 * kWidePsStride;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = j * 8 + 2 * c + (e & 1), t = tq * 16 + g + 8 * (e >> 1);
          pq[row * kWidePsStride + t] = s[j][e];
        }
    }
    if (wide_bar_or(!ok)) {
      ok = false;
      break;
    }

    // ---- B: rows warp and warp + 8, tokens 2 lane and 2 lane + 1
    const int tile0 = it.tok0 + n * kWideTok;
    const int nvalid = min(kWideTok, it.tok1 - tile0);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = warp + 8 * h;
      const float* pr = ps + r * kWidePsStride + 2 * lane;
      const float2 u = *reinterpret_cast<const float2*>(pr);
      const float2 v = *reinterpret_cast<const float2*>(pr + 16 * kWidePsStride);
      float x[2] = {u.x + v.x, u.y + v.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tt = 2 * lane + e, j = tile0 + tt;
        float y = x[e] * P.scale_log2;
        if (P.mask_type == PA_MASK_ALIBI) {
          y += slope2[h] * float(j - prow[h]);
        } else if (P.mask_type == PA_MASK_NORM_COMPRESS) {
          if (tt < nvalid && j > prow[h]) {  // above the diagonal only
            const int mr = min(max(prow[h] - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
            const int mc = min(max(j - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
            y += __half2float(P.mask[mr * PA_COMPRESS_MASK_SIZE + mc]) * kLog2e;
          }
        } else if (P.mask_type == PA_MASK_NORM) {
          if (tt < nvalid) y += norm_mask_log2(P, it.b, prow[h] - prefix, j);
        }
        x[e] = tt < nvalid ? y : -INFINITY;
      }
      const float mt = warp_max(fmaxf(x[0], x[1]));
      const float mn = fmaxf(m_run[h], mt);
      const float alpha = mn == m_run[h] ? 1.f : ex2(m_run[h] - mn);
      const float p0 = x[0] == -INFINITY ? 0.f : ex2(x[0] - mn);
      const float p1 = x[1] == -INFINITY ? 0.f : ex2(x[1] - mn);
      l_lane[h] = l_lane[h] * alpha + (p0 + p1);
      m_run[h] = mn;
      *reinterpret_cast<uint32_t*>(p_s + r * 128 + (((lane >> 2) ^ (r & 7)) << 4) + (lane & 3) * 4) =
          pack_half2(p0, p1);
      if (lane == 0) alpha_s[r] = alpha;
    }
    if (nvalid < kWideTok) {
      // Tokens past the range carry p = 0, but their V rows may hold anything
      // (stale or never-written shared memory, NaN included): zero them.
      const int rows = kWideTok - nvalid;
      for (int idx = tid; idx < VH * rows * 8; idx += NTH) {
        const int h = idx / (rows * 8), rem = idx % (rows * 8);
        const int t = nvalid + rem / 8, ch = rem % 8;
        *reinterpret_cast<uint4*>(tile + h * kWideHalfBytes + t * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      }
    }
    if (wide_bar_or(false)) break;  // P, alpha and the zeroed rows visible to all

    // ---- C: O^T (dims vd0..) *= alpha, += V^T P^T
    {
      const float a0 = alpha_s[2 * c], a1 = alpha_s[2 * c + 1];
      const float a2 = alpha_s[8 + 2 * c], a3 = alpha_s[8 + 2 * c + 1];
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt) {
        o[mt][0][0] *= a0;
        o[mt][0][1] *= a1;
        o[mt][0][2] *= a0;
        o[mt][0][3] *= a1;
        o[mt][1][0] *= a2;
        o[mt][1][1] *= a3;
        o[mt][1][2] *= a2;
        o[mt][1][3] *= a3;
      }
      const uint8_t* vb = tile + vh * kWideHalfBytes + v_row;
      const uint8_t* pb = p_s + p_row;
#pragma unroll
      for (int kk = 0; kk < kWideTok / 16; ++kk) {
        uint32_t b[4];
        ldsm_x4(b, pb + ((p_chk ^ uint32_t(2 * kk)) << 4));
        uint32_t va[MTW][4];
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt)
          ldsm_x4_t(va[mt], vb + kk * 2048 + ((v_chk ^ uint32_t(2 * mt)) << 4));
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt) {
          mma_16816(o[mt][0], va[mt], b[0], b[1]);
          mma_16816(o[mt][1], va[mt], b[2], b[3]);
        }
      }
    }
    // The slot returns to the producer once every warp is past its PV; P and
    // zeroed rows were written into it by threads, TMA refills it.
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }

  launch_dependents();  // the combine pass may be scheduled now

  // ---- epilogue: row sums, then O^T / l
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float l_row = warp_sum(l_lane[h]);
    if (lane == 0) {
      l_s[warp + 8 * h] = l_row;
      m_s[warp + 8 * h] = m_run[h];
    }
  }
  if (wide_bar_or(!ok)) {
    if (tid == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    return;
  }
  const bool partial = it.slot >= 0;
  if (partial && int64_t(it.slot) + it.nrows > P.part_rows_cap) {
    if (tid == 0) set_status(P.status, PA_STATUS_BIT_WORKSPACE);
    return;
  }
  if (ntiles == 0) {
    // an empty split (causal trim): weight zero in the combine
    if (partial)
      for (int idx = tid; idx < it.nrows * HV; idx += NTH) {
        P.part_o[int64_t(it.slot) * HV + idx] = __float2half_rn(0.f);
        if (idx % HV == 0) P.part_lse[it.slot + idx / HV] = -INFINITY;
      }
    return;
  }
  if (partial && tid < it.nrows) P.part_lse[it.slot + tid] = (m_s[tid] + log2f(l_s[tid])) * kLn2;
  float inv[2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) inv[j][e] = 1.f / l_s[j * 8 + 2 * c + e];
#pragma unroll
  for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = j * 8 + 2 * c + (e & 1);
        if (row >= it.nrows) continue;
        const int d = vd0 + mt * 16 + g + 8 * (e >> 1);
        const float val = o[mt][j][e] * inv[j][e & 1];
        if (partial) {
          P.part_o[(int64_t(it.slot) + row) * HV + d] = __float2half_rn(val);
        } else {
          const int rr = it.r0 + row;
          P.out[(int64_t(it.q_start + rr / G) * P.num_heads + it.kvh * G + rr % G) * HV + d] =
              __float2half_rn(val);
        }
      }
}

cudaError_t launch_wide(const CUtensorMap& tmk, const FwdParams& P, int64_t n_items,
                        cudaStream_t stream);

}  // namespace pa
