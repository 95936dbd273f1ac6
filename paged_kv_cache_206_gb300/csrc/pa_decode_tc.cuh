// Split-KV paged decode on the 5th-generation tensor cores (tcgen05 + TMEM) for
// 64-row query tiles: a wide GQA/MQA group (e.g. 64 query heads sharing one kv
// head of 512 dims, the shape of SparseAttnSharedkvMetadata's operator) makes
// QK^T and PV real dense tiles. PagedAttentionOperation semantics (block
// tables, context lengths, mask/bias); split/merge as in the metadata page.
//
// One CTA per work item, 6 warps:
//   warp 0     TMA producer: 128-token x 64-dim boxes (16 KB, 128-byte swizzle)
//              of K then V of each 128-token tile into a ring of 8 slots.
//   warp 1     allocates TMEM; one thread issues the MMAs:
//                S^T[128 tok x 64 rows]  = K . Q^T           (A, B K-major)
//                O^T[hv x 64 rows]      += V^T . P^T         (A, B MN-major)
//              with S^T and O^T accumulated in TMEM (fp32).
//   warps 2-5  softmax: thread = token (TMEM lane), its 64 scores in registers;
//              row max and row sum across the 128 tokens by a butterfly
//              reduce-scatter in each warp plus a 4-warp exchange in shared
//              memory; P^T (fp16) written to shared memory in the MN-major
//              swizzled layout the PV MMA reads; O^T rescaled in TMEM only when
//              a row's reference max must grow by more than 2^8 (exact: the
//              final normalisation uses the same reference); then the epilogue
//              (thread = output dim) reads O^T from TMEM and writes the rows.
// Every wait is bounded; on a timeout the CTA records PA_STATUS_BIT_TIMEOUT,
// lets its copies land, frees its TMEM and exits.
#pragma once

#include "pa_device.cuh"
#include "pa_warp_pipe.cuh"

namespace pa {

constexpr int kTcRows = PA_TC_TILE_ROWS;  // N of both MMAs (query rows, padded)
constexpr int kTcTok = 128;               // M of QK^T: tokens per tile
constexpr int kTcSlots = 8;               // ring of 16 KB boxes
constexpr uint32_t kTcSlotBytes = kTcTok * 128;  // 128 tokens x 64 dims x 2 B
constexpr int kTcThreads = 192;
constexpr float kTcRescaleThreshold = 8.f;  // log2 units

struct TcLayout {
  uint32_t q_off, p_off, ring_off, red_off, rows_off, bars_off, tmem_slot_off, bytes;
};

__host__ __device__ inline TcLayout tc_layout(int hk) {
  TcLayout L;
  L.q_off = 0;                                          // [hk/64][64 rows][128 B]
  L.p_off = L.q_off + uint32_t(hk / 64) * kTcRows * 128;  // [128 tok][64 rows] fp16
  L.ring_off = L.p_off + kTcTok * 128;                  // kTcSlots x 16 KB
  L.red_off = L.ring_off + kTcSlots * kTcSlotBytes;     // [4 warps][64] fp32 exchange
  L.rows_off = L.red_off + 4 * kTcRows * 4;             // per-row constants
  L.bars_off = L.rows_off + 6 * kTcRows * 4;            // mbarriers
  L.tmem_slot_off = L.bars_off + (2 * kTcSlots + 4) * 8;
  L.bytes = L.tmem_slot_off + 16 + 1024;
  return L;
}

// Head-size pairs the tcgen05 kernel is instantiated for (K boxes are consumed
// one 64-dim box at a time, V boxes in adjacent pairs of 128 dims).
inline bool tc_supported(int hk, int hv) {
  return hk == hv && (hk == 128 || hk == 256 || hk == 512);
}

// ---- tcgen05 / TMEM primitives --------------------------------------------

// Shared-memory matrix descriptor: 128-byte swizzle, version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((addr >> 4) & 0x3fff);
  d |= uint64_t((lbo >> 4) & 0x3fff) << 16;
  d |= uint64_t((sbo >> 4) & 0x3fff) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp16 A and B, fp32 D, M x N, majorness.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// Arrive once on `bar` when every previously issued tcgen05 op of this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive columns of this warp's TMEM lane quarter, written
// straight into v[0..32); the values may be read only after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]),
        "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]),
        "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]), "=f"(v[25]),
        "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barrier among the 128 softmax threads (warps 2-5).
__device__ __forceinline__ void softmax_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// The same barrier, returning the OR of `pred` over the 128 threads: every
// softmax thread takes the same continue/abort decision.
__device__ __forceinline__ bool softmax_bar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(uint32_t(pred))
      : "memory");
  return r != 0;
}

// Lane 0 waits; the whole warp gets its verdict.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane) {
  bool ok = true;
  if (lane == 0) ok = mbar_wait(bar, parity);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Butterfly reduce-scatter of v[64] (one value per row) across the warp:
// afterwards lane l holds the reduction of rows 2l and 2l+1 in v[0], v[1].
template <bool MAX>
__device__ __forceinline__ void reduce_scatter64(float (&v)[64], int lane) {
#pragma unroll
  for (int lvl = 0; lvl < 5; ++lvl) {
    const int off = 16 >> lvl;
    const int half = 32 >> lvl;  // values kept after this level
    const bool upper = lane & off;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, off);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

template <int HK, int HV>
__global__ void __launch_bounds__(kTcThreads, 1) tc_decode_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
    const FwdParams P) {
  constexpr int KB = HK / 64;   // K boxes (slots) per tile
  constexpr int VB = HV / 64;   // V boxes per tile, consumed in pairs
  constexpr int OC = HV / 128;  // O^T chunks of 128 dims
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdescQK = mma_idesc(128, kTcRows, 0, 0);
  constexpr uint32_t kIdescPV = mma_idesc(128, kTcRows, 1, 1);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  const TcLayout lay = tc_layout(HK);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* q_s = smem + lay.q_off;
  uint8_t* p_s = smem + lay.p_off;
  uint8_t* ring = smem + lay.ring_off;
  float* red = reinterpret_cast<float*>(smem + lay.red_off);
  float* m_used = reinterpret_cast<float*>(smem + lay.rows_off);  // [64] reference max (base 2)
  float* alpha_s = m_used + kTcRows;                              // [64] rescale factors
  float* slope2 = alpha_s + kTcRows;                              // [64]
  int* prow = reinterpret_cast<int*>(slope2 + kTcRows);           // [64]
  float* l_tot = slope2 + 2 * kTcRows;                            // [64]
  int* flags = reinterpret_cast<int*>(l_tot + kTcRows);           // [1] rescale this tile
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars_off);
  uint64_t* empty = full + kTcSlots;
  uint64_t* s_full = empty + kTcSlots;
  uint64_t* p_full = s_full + 1;
  uint64_t* o_done = s_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + lay.tmem_slot_off);

  Item it;
  it.load(P, blockIdx.x);
  const int G = P.group, bs = P.block_size;
  const int ntok = it.tok1 - it.tok0;
  const int ntiles = ntok > 0 ? (ntok + kTcTok - 1) / kTcTok : 0;
  const int prefix = it.L - it.qlen;
  const int sigma = it.L > PA_COMPRESS_MASK_SIZE ? it.L - PA_COMPRESS_MASK_SIZE : 0;

  // ---- set-up: barriers, TMEM, query tile, per-row constants
  if (tid == 0) {
    for (int s = 0; s < kTcSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    fence_barrier_init();
    flags[1] = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // Q tile: row r of the tile, chunk c (8 dims) -> box c/8, swizzled position.
  for (int idx = tid; idx < kTcRows * (HK / 8); idx += kTcThreads) {
    const int r = idx / (HK / 8), c = idx % (HK / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < it.nrows) {
      const int rr = it.r0 + r;
      v = *reinterpret_cast<const uint4*>(
          P.query + (int64_t(it.q_start + rr / G) * P.num_heads + it.kvh * G + rr % G) * HK + c * 8);
    }
    *reinterpret_cast<uint4*>(q_s + (c >> 3) * (kTcRows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
  }
  for (int r = tid; r < kTcRows; r += kTcThreads) {
    const bool ok = r < it.nrows;
    const int rr = it.r0 + r;
    prow[r] = ok ? prefix + rr / G : it.L - 1;
    slope2[r] = (ok && P.mask_type == PA_MASK_ALIBI) ? P.alibi_slopes[it.kvh * G + rr % G] * kLog2e : 0.f;
    m_used[r] = -INFINITY;
    l_tot[r] = 0.f;
  }
  fence_proxy_async();  // query tile written by threads, read by the tensor cores
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem;        // S^T: columns [0, 64)
  const uint32_t tmem_o = tmem + 64;   // O^T chunk c: columns [64 + 64 c, 128 + 64 c)

  if (warp == 0) {
    // ================= TMA producer (lane 0) =================
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int32_t* bt_row = P.block_tables + int64_t(it.b) * P.max_blocks_per_seq;
      const int box_rows = bs < kTcTok ? bs : kTcTok;
      const int pieces = kTcTok / box_rows;
      int issued = 0;
      bool ok = true;
      for (int n = 0; n < ntiles && ok; ++n) {
        const int t0 = it.tok0 + n * kTcTok;  // first token of the tile
        for (int part = 0; part < KB + VB; ++part) {
          const int slot = issued % kTcSlots;
          if (!mbar_wait(&empty[slot], ((issued / kTcSlots) & 1) ^ 1)) {
            ok = false;
            break;
          }
          const bool is_k = part < KB;
          const int box = is_k ? part : part - KB;
          uint8_t* dst = ring + slot * kTcSlotBytes;
          // pieces of box_rows tokens from consecutive blocks; those past the
          // range are not loaded (their rows are masked or zeroed later)
          uint32_t bytes = 0;
          int phys[8];
          for (int pc = 0; pc < pieces; ++pc) {
            const int tok = t0 + pc * box_rows;
            phys[pc] = -1;
            if (tok < it.tok1) {
              const int ph = bt_row[tok / bs];
              if (ph < 0 || ph >= P.num_blocks) {
                set_status(P.status, PA_STATUS_BIT_BLOCK_INDEX);
              } else {
                phys[pc] = ph;
                bytes += uint32_t(box_rows) * 128;
              }
            }
          }
          if (bytes) {
            mbar_arrive_expect_tx(&full[slot], bytes);
          } else {
            mbar_arrive(&full[slot]);
          }
          for (int pc = 0; pc < pieces; ++pc) {
            if (phys[pc] < 0) continue;
            const int tok = t0 + pc * box_rows;
            const int row = phys[pc] * bs + tok % bs;
            tma_load_2d(dst + pc * box_rows * 128, is_k ? &tmk : &tmv, &full[slot],
                        it.kvh * (is_k ? HK : HV) + box * 64, row, pol);
          }
          ++issued;
        }
      }
      if (!ok) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
      // let every issued copy land before the CTA can exit (bounded waits)
      for (int i = issued - kTcSlots > 0 ? issued - kTcSlots : 0; i < issued; ++i)
        mbar_wait(&full[i % kTcSlots], (i / kTcSlots) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer =================
    int consumed = 0;
    bool ok = true;
    const uint32_t q_addr = smem_u32(q_s), p_addr = smem_u32(p_s), ring_addr = smem_u32(ring);
    for (int n = 0; n < ntiles && ok; ++n) {
      // S^T = K . Q^T over the KB boxes of 64 dims (4 k-steps of 16 each)
      for (int kb = 0; kb < KB; ++kb, ++consumed) {
        const int slot = consumed % kTcSlots;
        if (!warp_wait(&full[slot], (consumed / kTcSlots) & 1, lane)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t a = smem_desc(ring_addr + slot * kTcSlotBytes + k * 32, 16, 1024);
            const uint64_t b = smem_desc(q_addr + kb * (kTcRows * 128) + k * 32, 16, 1024);
            tc_mma(tmem_s, a, b, kIdescQK, (kb | k) != 0);
          }
          tc_commit(&empty[slot]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(s_full);
      __syncwarp();
      // O^T += V^T . P^T once the softmax has written P^T
      if (!warp_wait(p_full, n & 1, lane)) { ok = false; break; }
      tc_fence_after();
      const int nvalid = min(kTcTok, it.tok1 - (it.tok0 + n * kTcTok));
      for (int oc = 0; oc < OC; ++oc, consumed += 2) {
        const int s0 = consumed % kTcSlots, s1 = (consumed + 1) % kTcSlots;
        if (!warp_wait(&full[s0], (consumed / kTcSlots) & 1, lane) ||
            !warp_wait(&full[s1], ((consumed + 1) / kTcSlots) & 1, lane)) { ok = false; break; }
        if (nvalid < kTcTok) {
          // V rows of tokens past the range may hold anything (NaN included):
          // zero them so that p = 0 really contributes nothing.
          for (int idx = lane; idx < (kTcTok - nvalid) * 8 * 2; idx += 32) {
            const int sl = idx / ((kTcTok - nvalid) * 8) ? s1 : s0;
            const int rem = idx % ((kTcTok - nvalid) * 8);
            *reinterpret_cast<uint4*>(ring + sl * kTcSlotBytes + (nvalid + rem / 8) * 128 +
                                      (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
          // the pair of boxes is adjacent only when s1 == s0 + 1 (slots are
          // consumed in pairs from an even index, and the ring size is even)
#pragma unroll
          for (int k = 0; k < kTcTok / 16; ++k) {
            const uint64_t a = smem_desc(ring_addr + s0 * kTcSlotBytes + k * 2048, kTcSlotBytes, 1024);
            const uint64_t b = smem_desc(p_addr + k * 2048, kTcSlotBytes, 1024);
            tc_mma(tmem_o + oc * 64, a, b, kIdescPV, (n | k) != 0);
          }
          tc_commit(&empty[s0]);
          tc_commit(&empty[s1]);
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    if (lane == 0) tc_commit(o_done);  // completes when every MMA above is done
    __syncwarp();
  } else {
    // ================= softmax warps 2-5 =================
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int t = quarter * 32 + lane;        // token within the tile (= TMEM lane)
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    float l_part[2] = {0.f, 0.f};             // row sums of rows 2*lane, 2*lane+1 (this warp)
    bool ok = true;
    for (int n = 0; n < ntiles; ++n) {
      const bool got = mbar_wait(s_full, n & 1);
      if (softmax_bar_or(!got)) { ok = false; break; }  // all four warps agree
      tc_fence_after();
      float s[64];
      tmem_ld32(tmem_s + lane_base, s);
      tmem_ld32(tmem_s + lane_base + 32, s + 32);
      tmem_wait_ld();
      const int j = it.tok0 + n * kTcTok + t;
      const bool tok_ok = j < it.tok1;
#pragma unroll
      for (int r = 0; r < 64; ++r) {
        float v = s[r] * P.scale_log2;
        if (P.mask_type == PA_MASK_ALIBI) {
          v += slope2[r] * float(j - prow[r]);
        } else if (P.mask_type == PA_MASK_NORM_COMPRESS) {
          if (tok_ok && j > prefix) {
            const int mr = min(max(prow[r] - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
            const int mc = min(max(j - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
            v += __half2float(P.mask[mr * PA_COMPRESS_MASK_SIZE + mc]) * kLog2e;
          }
        }
        s[r] = tok_ok ? v : -INFINITY;
      }
      // tile max per row: reduce-scatter in the warp, then across the 4 warps
      float w[64];
#pragma unroll
      for (int r = 0; r < 64; ++r) w[r] = s[r];
      reduce_scatter64<true>(w, lane);
      red[quarter * 64 + 2 * lane] = w[0];
      red[quarter * 64 + 2 * lane + 1] = w[1];
      softmax_bar();
      if (warp == 2) {
        // reference max update for rows 2*lane, 2*lane+1 (lazy rescale)
        bool grow = false;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = 2 * lane + e;
          const float mt = fmaxf(fmaxf(red[r], red[64 + r]), fmaxf(red[128 + r], red[192 + r]));
          const float mu = m_used[r];
          float a = 1.f;
          if (mt > mu + kTcRescaleThreshold || mu == -INFINITY) {
            const float nm = fmaxf(mt, mu);
            a = ex2(mu - nm);  // 0 on the first tile
            m_used[r] = nm;
            grow = grow || (mu != -INFINITY);
          }
          alpha_s[r] = a;
        }
        grow = __any_sync(0xffffffffu, grow);
        if (lane == 0) flags[1] = grow ? 1 : 0;
      }
      softmax_bar();
      const bool rescale = flags[1] != 0;
      if (rescale) {
        // O^T rows of this thread's TMEM lane (= output dims) times alpha per column;
        // PV of the previous tile is complete: S^T of this tile was committed after it.
        l_part[0] *= alpha_s[2 * lane];
        l_part[1] *= alpha_s[2 * lane + 1];
#pragma unroll 1
        for (int oc = 0; oc < OC; ++oc) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float o[32];
            const uint32_t ta = tmem_o + oc * 64 + h * 32 + lane_base;
            tmem_ld32(ta, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha_s[h * 32 + i];
            tmem_st32(ta, o);
          }
        }
        tmem_wait_st();
      }
      // probabilities, row sums, P^T into shared memory (token row t, 64 rows of fp16)
#pragma unroll
      for (int r = 0; r < 64; ++r) s[r] = ex2(s[r] - m_used[r]);
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint4 pk;
        pk.x = pack_half2(s[c8 * 8 + 0], s[c8 * 8 + 1]);
        pk.y = pack_half2(s[c8 * 8 + 2], s[c8 * 8 + 3]);
        pk.z = pack_half2(s[c8 * 8 + 4], s[c8 * 8 + 5]);
        pk.w = pack_half2(s[c8 * 8 + 6], s[c8 * 8 + 7]);
        *reinterpret_cast<uint4*>(p_s + t * 128 + ((c8 ^ (t & 7)) << 4)) = pk;
      }
      reduce_scatter64<false>(s, lane);
      l_part[0] += s[0];
      l_part[1] += s[1];
      fence_proxy_async();  // P^T is read by the tensor cores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (!ok && t == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    // ---- epilogue: row sums across the 4 warps, then O^T / l
    red[quarter * 64 + 2 * lane] = l_part[0];
    red[quarter * 64 + 2 * lane + 1] = l_part[1];
    softmax_bar();
    if (warp == 2) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = 2 * lane + e;
        l_tot[r] = (red[r] + red[64 + r]) + (red[128 + r] + red[192 + r]);
      }
    }
    launch_dependents();
    const bool got = ok && mbar_wait(o_done, 0);
    const bool done = !softmax_bar_or(!got);
    if (done && ntiles > 0) {
      tc_fence_after();
      const bool partial = it.slot >= 0;
      const bool fits = !partial || int64_t(it.slot) + it.nrows <= P.part_rows_cap;
      if (!fits && t == 0) set_status(P.status, PA_STATUS_BIT_WORKSPACE);
#pragma unroll 1
      for (int oc = 0; oc < OC; ++oc) {
        const int d = oc * 128 + t;  // output dim of this thread
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float o[32];
          tmem_ld32(tmem_o + oc * 64 + h * 32 + lane_base, o);
          tmem_wait_ld();
          if (!fits) continue;
#pragma unroll 4
          for (int i = 0; i < 32; ++i) {
            const int r = h * 32 + i;
            if (r >= it.nrows) break;
            const float val = o[i] / l_tot[r];
            if (!partial) {
              const int rr = it.r0 + r;
              P.out[(int64_t(it.q_start + rr / G) * P.num_heads + it.kvh * G + rr % G) * HV + d] =
                  __float2half_rn(val);
            } else {
              P.part_o[(int64_t(it.slot) + r) * HV + d] = val;
              if (d == 0) P.part_lse[it.slot + r] = (m_used[r] + log2f(l_tot[r])) * kLn2;
            }
          }
        }
      }
    }
  }
  // ---- teardown: every tcgen05 op has completed (o_done) before TMEM is freed
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) mbar_wait(o_done, 0);
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols));
  }
}

cudaError_t launch_tc(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                      int64_t n_items, cudaStream_t stream);

}  // namespace pa
