// Split-KV paged decode on the 5th-generation tensor cores (tcgen05 + TMEM) for
// 64-row query tiles: a wide GQA/MQA group (e.g. 64 query heads sharing one kv
// head of 512 dims, the shape of SparseAttnSharedkvMetadata's operator) makes
// QK^T and PV real dense tiles. PagedAttentionOperation semantics (block
// tables, context lengths, mask/bias); split/merge as in the metadata page.
//
// The KV range of a work item is cut into 64-token tiles. One CTA per item,
// 12 warps:
//   warp 0     K producer: 3-D TMA boxes of 64 tokens x 128 dims (16 KB, two
//              128-byte-swizzled 64-dim halves) into the K ring.
//   warp 10    V producer: the same for V into the V ring (ring sizes: TcCfg,
//              from the shared memory the query tile leaves, e.g. 5 K + 4 V
//              slots at 512 dims and 64 rows).
//   warp 1     allocates TMEM; one thread issues S^T[64 tok x 64 rows] = K . Q^T
//              (M=64; A, B K-major) into one of two S^T buffers in TMEM, up to
//              two tiles ahead of the softmax.
//   warp 11    one thread issues O^T[hv x 64 rows] += V^T . P^T (M=128; A, B
//              MN-major) as soon as a tile's P^T is ready; O^T stays in TMEM.
//   warps 2-9  softmax: two warps per TMEM lane quarter; with M=64 a quarter
//              holds 16 tokens (lanes 0-15), and each warp of the pair takes 32
//              of the 64 rows. Probabilities are taken against a per-row
//              reference max that is recomputed exactly (warp max + 4-quarter
//              exchange) only when some score exceeds it by more than 2^8 -- in
//              practice the first tile; O^T and the sums are rescaled then
//              (exact: the final normalisation uses the same reference). Row
//              sums accumulate per token and are reduced across tokens once, at
//              the end. P^T (fp16) goes to shared memory in the MN-major
//              swizzled layout the PV MMA reads. Epilogue: thread = output dim,
//              O^T / l from TMEM to the output or the split partials.
// Separate rings and issuers keep K streaming into QK while a tile's V waits
// for its softmax. Every wait is bounded; on a timeout the CTA records
// PA_STATUS_BIT_TIMEOUT, lets its copies land, frees its TMEM and exits.
#pragma once

#include "pa_device.cuh"
#include "pa_warp_pipe.cuh"

namespace pa {

constexpr int kTcRows = PA_TC_TILE_ROWS;  // rows of a tile at most; N of the PV MMA
constexpr int kTcTok = 64;                // tokens per tile (M of QK^T)
constexpr int kTcPBufs = 1;               // P^T buffers of separate caches (softmax of tile
                                          // n + kTcPBufs waits for the PV of tile n)
constexpr uint32_t kTcMaxSmem = 232448;   // dynamic shared memory a CTA may use
constexpr uint32_t kTcHalfBytes = kTcTok * 128;      // 64 tokens x 64 dims x 2 B
constexpr uint32_t kTcSlotBytes = 2 * kTcHalfBytes;  // 64 tokens x 128 dims
constexpr int kTcThreads = 384;  // 2 producers, 2 MMA issuers, 8 softmax warps
constexpr float kTcRescaleThreshold = 8.f;  // log2 units

// Shared-memory plan of a launch with NR query rows per tile (16, 32 or 64:
// the group's rows G * max_q rounded up): the query tile [hk/64][NR][128 B],
// P^T [64 tokens][64 rows] (rows past NR stay zero), the K ring, the V ring,
// the row exchange and constants, the barriers. The rings take what the query
// tile leaves, at most 12 slots of 16 KB, split between K and V (K gets the
// odd one: a sweep over ring sizes found K the more sensitive). With a
// shared-KV cache (SH) there is no V ring: the PV MMAs read V from the K
// slots, which then stay until the tile's PV is done, and every slot is K's.
template <int HK, int NR, bool SH = false>
struct TcCfg {
  static constexpr uint32_t kQBytes = uint32_t(HK / 64) * NR * 128;
  // The shared 576/512 cache is paced by the MMA issue: a second P^T buffer
  // (one K slot less) lets the softmax of tile n + 1 run under the PV of tile n.
  static constexpr int kPBufs = SH ? 2 : kTcPBufs;
  static constexpr uint32_t kOther = kPBufs * kTcTok * 128 + 4 * kTcRows * 4 +
                                     6 * kTcRows * 4 + 12 * 8 + 16 + 1024;
  static constexpr int kFit = int((kTcMaxSmem - kQBytes - kOther) / (kTcSlotBytes + 16));
  static constexpr int kSlots = kFit < 12 ? kFit : 12;
  static constexpr int kKSlots = SH ? kSlots : (kSlots + 1) / 2;
  static constexpr int kVSlots = SH ? 0 : kSlots / 2;
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t p_off = q_off + kQBytes;
  static constexpr uint32_t ring_off = p_off + kPBufs * kTcTok * 128;  // 1024-aligned
  static constexpr uint32_t red_off = ring_off + kSlots * kTcSlotBytes;  // [4][64] fp32
  static constexpr uint32_t rows_off = red_off + 4 * kTcRows * 4;        // per-row constants
  static constexpr uint32_t bars_off = rows_off + 6 * kTcRows * 4;       // mbarriers
  static constexpr uint32_t tmem_slot_off = bars_off + (2 * kSlots + 12) * 8;
  static constexpr uint32_t bytes = tmem_slot_off + 16 + 1024;
  static_assert(kKSlots >= 4 && (SH || kVSlots >= 4), "rings of at least one tile");
  static_assert(!SH || kKSlots >= (HK / 64 + 1) / 2, "a shared-KV ring holds a whole tile");
  static_assert(bytes <= kTcMaxSmem, "shared memory");
};

// Head-size pairs the tcgen05 kernel is instantiated for (K and V move in
// 16 KB slots of 64 tokens x 128 dims; a 576-dim K row takes four and a half).
inline bool tc_supported(int hk, int hv) {
  return (hk == hv && (hk == 128 || hk == 256 || hk == 512)) || (hk == 576 && hv == 512);
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

// RH (8, 16 or 32) consecutive columns of this warp's TMEM lane quarter.
template <int RH>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v) {
  if constexpr (RH == 32) {
    tmem_ld32(taddr, v);
  } else if constexpr (RH == 16) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
        : "r"(taddr)
        : "memory");
  } else {
    static_assert(RH == 8, "8, 16 or 32 columns");
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                   "=f"(v[6]), "=f"(v[7])
                 : "r"(taddr)
                 : "memory");
  }
}

template <int RH>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float* v) {
  if constexpr (RH == 32) {
    tmem_st32(taddr, *reinterpret_cast<const float(*)[32]>(v));
  } else if constexpr (RH == 16) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
  } else {
    static_assert(RH == 8, "8, 16 or 32 columns");
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
        : "memory");
  }
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barrier among the 256 softmax threads (warps 2-9).
__device__ __forceinline__ void softmax_bar() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// The same barrier, returning the OR of `pred` over the 256 threads: every
// softmax thread takes the same continue/abort decision.
__device__ __forceinline__ bool softmax_bar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(uint32_t(pred))
      : "memory");
  return r != 0;
}

// Lane 0 waits; the whole warp gets its verdict.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane,
                                          long long limit = kWaitLimitCycles) {
  bool ok = true;
  if (lane == 0) ok = mbar_wait(bar, parity, limit);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <int HK, int HV, int NR, bool SH>
__global__ void __launch_bounds__(kTcThreads, 1) tc_decode_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
    const __grid_constant__ CUtensorMap tmq, const FwdParams P) {
  constexpr int KH = HK / 64;         // 64-dim halves of a K row
  constexpr int KS = (KH + 1) / 2;    // K slots per tile (128 dims each; the
                                      // last holds one half when KH is odd)
  constexpr int VS = HV / 128;  // V slots per tile = O^T chunks of 128 dims
  constexpr uint32_t kTmemCols = 512;
  using Cfg = TcCfg<HK, NR, SH>;
  constexpr int kKSlots = Cfg::kKSlots, kVSlots = Cfg::kVSlots;
  constexpr int PB = Cfg::kPBufs;
  constexpr int RH = NR / 2;  // rows per softmax thread (two warps per lane quarter)
  constexpr uint32_t kIdescQK = mma_idesc(64, NR, 0, 0);
  // PV reads the first NR columns of each 128-byte P^T row (the tile's rows)
  constexpr uint32_t kIdescPV = mma_idesc(128, NR, 1, 1);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* q_s = smem + Cfg::q_off;
  uint8_t* p_s = smem + Cfg::p_off;
  uint8_t* kring = smem + Cfg::ring_off;
  uint8_t* vring = kring + kKSlots * kTcSlotBytes;
  float* red = reinterpret_cast<float*>(smem + Cfg::red_off);
  float* m_used = reinterpret_cast<float*>(smem + Cfg::rows_off);  // [64] reference max (base 2)
  float* alpha_s = m_used + kTcRows;                              // [64] rescale factors
  float* slope2 = alpha_s + kTcRows;                              // [64]
  int* prow = reinterpret_cast<int*>(slope2 + kTcRows);           // [64]
  float* l_tot = slope2 + 2 * kTcRows;                            // [64]
  int* flags = reinterpret_cast<int*>(l_tot + kTcRows);           // [1] rescale this tile
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + Cfg::bars_off);
  uint64_t* kempty = kfull + kKSlots;
  uint64_t* vfull = kempty + kKSlots;
  uint64_t* vempty = vfull + kVSlots;
  uint64_t* s_full = vempty + kVSlots;  // [2] S^T buffer ready
  uint64_t* s_free = s_full + 2;          // [2] S^T buffer read by every softmax warp
  uint64_t* p_full = s_full + 4;          // [2] P^T buffer written
  uint64_t* pv_done = s_full + 6;         // [2] PV that read P^T buffer b complete
  uint64_t* qk_done = s_full + 8;         // every QK MMA complete
  uint64_t* o_done = s_full + 9;          // every PV MMA complete
  uint64_t* q_ready = s_full + 10;        // query tile in shared memory (one arrival per softmax warp)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::tmem_slot_off);

  if (P.counts && int(blockIdx.x) >= P.counts[0]) return;  // past a device plan's items
  Item it;
  it.load(P, blockIdx.x);
  const int G = P.group, bs = P.block_size;
  const int prefix = it.L - it.qlen;
  if (P.mask_type == PA_MASK_NORM_COMPRESS && it.nrows > 0) {
    // Causal trim: keys past the position of the tile's last query token are
    // masked (a large negative fill) for every row of the tile, so their
    // probabilities are exactly zero in fp32; the item stops before them.
    // Prefill tiles (q = L) thus skip the upper triangle; a split that lies
    // wholly past it becomes empty (never split 0, which starts at key 0).
    const int pmax = prefix + (it.r0 + it.nrows - 1) / G;
    it.tok1 = max(it.tok0, min(it.tok1, pmax + 1));
  }
  const int ntok = it.tok1 - it.tok0;
  const int ntiles = ntok > 0 ? (ntok + kTcTok - 1) / kTcTok : 0;
  const int sigma = it.L > PA_COMPRESS_MASK_SIZE ? it.L - PA_COMPRESS_MASK_SIZE : 0;

  // ---- set-up: barriers, TMEM, query tile, per-row constants
  if (tid == 0) {
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(&vfull[s], 1);
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
    mbar_init(q_ready, P.q_tma ? 9 : 8);  // + the producer's query copy
    fence_barrier_init();
    flags[1] = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  for (int r = tid; r < kTcRows; r += kTcThreads) {
    const bool ok = r < it.nrows;
    const int rr = it.r0 + r;
    prow[r] = ok ? prefix + rr / G : it.L - 1;
    slope2[r] = (ok && P.mask_type == PA_MASK_ALIBI) ? P.alibi_slopes[it.kvh * G + rr % G] * kLog2e : 0.f;
    m_used[r] = -INFINITY;
    l_tot[r] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem;        // S^T buffer b: columns [64 b, 64 b + 64)
  const uint32_t tmem_o = tmem + 128;  // O^T chunk c: columns [128 + 64 c, 192 + 64 c)

  if (warp == 0 || warp == 10) {
    // ================= TMA producers (lane 0): K (warp 0), V (warp 10) =========
    if (lane == 0 && !(SH && warp == 10)) {
      const bool is_k = warp == 0;
      const int nslots = is_k ? kKSlots : kVSlots;
      uint8_t* ring = is_k ? kring : vring;
      uint64_t* full = is_k ? kfull : vfull;
      uint64_t* empty = is_k ? kempty : vempty;
      const CUtensorMap* map = is_k ? &tmk : &tmv;
      const int per_tile = is_k ? KS : VS;
      // 64-dim blocks per kv head in the map's rows: a shared-KV V map spans the K rows
      const int zbase = it.kvh * ((is_k || P.kv_shared ? HK : HV) / 64);
      const uint64_t pol = policy_evict_first();
      // V copies start once the query tile has landed: the first QK (query
      // and K tile 0) is then not queued behind every CTA's V ring
      if (!is_k && P.q_tma && !mbar_wait(q_ready, 0, P.wait_limit)) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
      if (is_k && P.q_tma) {
        // The query tile first, ahead of the K ring in the same queue: its G
        // rows (heads kvh * G .. of the sequence's one query token) are
        // consecutive in the query; one box per 64-dim block (q_tma 1), or
        // one box of every block when the tile's rows are exactly the G
        // (q_tma 2), landing where the QK MMA reads it. Every split of the
        // tile reads the same tile, so keep it in L2.
        const int G = P.group;
        mbar_arrive_expect_tx(q_ready, uint32_t(KH) * G * 128);
        const int row0 = it.q_start * P.num_heads + it.kvh * G;
        if (P.q_tma == 2) {
          tma_load_3d(q_s, &tmq, q_ready, 0, row0, 0, policy_evict_last());
        } else {
          for (int blk = 0; blk < KH; ++blk)
            tma_load_3d(q_s + blk * (NR * 128), &tmq, q_ready, 0, row0, blk, policy_evict_last());
        }
      }
      const int32_t* bt_row = P.block_tables + int64_t(it.b) * P.max_blocks_per_seq;
      // the largest power of two dividing both the block and the tile: a
      // box never crosses a block (block_size 96 moves 32-token boxes)
      const int box_rows = (bs & -bs) < kTcTok ? (bs & -bs) : kTcTok;
      const int pieces = kTcTok / box_rows;
      int issued = 0;
      bool ok = true;
      for (int n = 0; n < ntiles && ok; ++n) {
        // physical rows of the tile's pieces (-1: past the range or a bad entry)
        const int t0 = it.tok0 + n * kTcTok;
        int ph[4], rws[4];
        for (int pc = 0; pc < pieces; ++pc) {
          const int tok = t0 + pc * box_rows;
          ph[pc] = tok < it.tok1 ? bt_row[tok / bs] : -1;
        }
        int npieces = 0;
        for (int pc = 0; pc < pieces; ++pc) {
          const int tok = t0 + pc * box_rows;
          rws[pc] = -1;
          if (tok >= it.tok1) continue;
          if (ph[pc] < 0 || ph[pc] >= P.num_blocks) {
            if (is_k) set_status(P.status, PA_STATUS_BIT_BLOCK_INDEX);
            continue;
          }
          rws[pc] = ph[pc] * bs + tok % bs;
          ++npieces;
        }
        for (int sl = 0; sl < per_tile; ++sl) {
          // the last K slot of an odd number of halves carries one half; a
          // 64-token box still moves two (the second is the next 64 dims of
          // the row, or the fill value past the tensor) and is left unread
          const bool one_half = is_k && (KH & 1) && sl == KS - 1 && box_rows != kTcTok;
          const uint32_t bytes = uint32_t(npieces) * box_rows * (one_half ? 128 : 256);
          const int slot = issued % nslots;
          if (!mbar_wait(&empty[slot], ((issued / nslots) & 1) ^ 1, P.wait_limit)) {
            ok = false;
            break;
          }
          uint8_t* dst = ring + slot * kTcSlotBytes;
          if (bytes) {
            mbar_arrive_expect_tx(&full[slot], bytes);
          } else {
            mbar_arrive(&full[slot]);
          }
          const int z = zbase + 2 * sl;  // first 64-dim half of this slot
          for (int pc = 0; pc < pieces; ++pc) {
            if (rws[pc] < 0) continue;
            if (box_rows == kTcTok) {
              // one box carries both halves: [2][64 tokens][128 B] = the slot
              tma_load_3d(dst, map, &full[slot], 0, rws[pc], z, pol);
            } else {
              // block_size < 64: the map's box is one half; place each half
              tma_load_3d(dst + pc * box_rows * 128, map, &full[slot], 0, rws[pc], z, pol);
              if (!one_half)
                tma_load_3d(dst + kTcHalfBytes + pc * box_rows * 128, map, &full[slot], 0,
                            rws[pc], z + 1, pol);
            }
          }
          ++issued;
        }
      }
      if (!ok) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
      // let every issued copy land before the CTA can exit (bounded waits,
      // default limit), the query tile's too
      for (int i = issued - nslots > 0 ? issued - nslots : 0; i < issued; ++i)
        mbar_wait(&full[i % nslots], (i / nslots) & 1);
      if (is_k && P.q_tma) mbar_wait(q_ready, 0);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= QK issuer =================
    if constexpr (SH) {
      // S^T(m) into buffer m & 1 once the softmax has read S^T(m - 2). Lane 0
      // alone waits and issues (a tcgen05.mma costs about 50 cycles to issue
      // whatever its shape, and the issue of these small ones is what paces a
      // narrow tile of the shared 576/512 cache): no warp-wide exchange per
      // slot. Separate caches keep the warp-wide form below.
      if (lane == 0) {
        bool ok = true;
        const uint32_t q_addr = smem_u32(q_s), ring_addr = smem_u32(kring);
        int consumed = 0;
        // the query tile (TMA or the softmax warps' loads) while the producers stream
        if (ntiles > 0 && !mbar_wait(q_ready, 0, P.wait_limit)) ok = false;
        for (int m = 0; m < ntiles && ok; ++m) {
          if (m >= 2 && !mbar_wait(&s_free[m & 1], ((m >> 1) - 1) & 1, P.wait_limit)) { ok = false; break; }
          tc_fence_after();
          for (int ks = 0; ks < KS; ++ks, ++consumed) {
            const int slot = consumed % kKSlots;
            if (!mbar_wait(&kfull[slot], (consumed / kKSlots) & 1, P.wait_limit)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (2 * ks + h >= KH) break;  // an odd KH leaves the last slot one half
              const uint64_t a = smem_desc(ring_addr + slot * kTcSlotBytes + h * kTcHalfBytes, 16, 1024);
              const uint64_t b = smem_desc(q_addr + (2 * ks + h) * (NR * 128), 16, 1024);
#pragma unroll
              for (int k = 0; k < 4; ++k)  // +32 bytes a k-step: +2 in the address field
                tc_mma(tmem_s + (m & 1) * 64, a + 2 * k, b + 2 * k, kIdescQK, (ks | h | k) != 0);
            }
            // (the slot is released after the PV: V is its first dims)
          }
          if (!ok) break;
          tc_commit(&s_full[m & 1]);
        }
        if (!ok) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
        tc_commit(qk_done);
      }
      __syncwarp();
    } else {
      // S^T(m) into buffer m & 1 once the softmax has read S^T(m - 2).
      bool ok = true;
      const uint32_t q_addr = smem_u32(q_s), ring_addr = smem_u32(kring);
      int consumed = 0;
      // the softmax warps load the query tile while the producers already stream
      if (ntiles > 0 && !warp_wait(q_ready, 0, lane, P.wait_limit)) ok = false;
      for (int m = 0; m < ntiles && ok; ++m) {
        if (m >= 2 && !warp_wait(&s_free[m & 1], ((m >> 1) - 1) & 1, lane, P.wait_limit)) { ok = false; break; }
        tc_fence_after();
        for (int ks = 0; ks < KS; ++ks, ++consumed) {
          const int slot = consumed % kKSlots;
          if (!warp_wait(&kfull[slot], (consumed / kKSlots) & 1, lane, P.wait_limit)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (2 * ks + h >= KH) break;  // an odd KH leaves the last slot one half
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t a = smem_desc(ring_addr + slot * kTcSlotBytes + h * kTcHalfBytes + k * 32, 16, 1024);
                const uint64_t b = smem_desc(q_addr + (2 * ks + h) * (NR * 128) + k * 32, 16, 1024);
                tc_mma(tmem_s + (m & 1) * 64, a, b, kIdescQK, (ks | h | k) != 0);
              }
            }
            tc_commit(&kempty[slot]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) tc_commit(&s_full[m & 1]);
        __syncwarp();
      }
      if (!ok && lane == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
      if (lane == 0) tc_commit(qk_done);
      __syncwarp();
    }
  } else if (warp == 11) {
    // ================= PV issuer =================
    // Shared-KV cache: lane 0 waits and issues a full tile alone, the whole
    // warp joining only on a tile with rows past the range, to zero them.
    // Separate caches keep the warp-wide waits (measured faster there: the
    // lane-0 form changed the register allocation of the 64-row kernel).
    bool ok = true;
    uint8_t* const ring = SH ? kring : vring;  // shared KV: V is in the K slots
    const uint32_t p_addr = smem_u32(p_s), ring_addr = smem_u32(ring);
    int consumed = 0;
    for (int n = 0; n < ntiles && ok; ++n) {
      const int pb = n % PB;
      const int nvalid = min(kTcTok, it.tok1 - (it.tok0 + n * kTcTok));
      if (SH && nvalid == kTcTok) {
        // a full tile. Shared KV: chunk oc is K slot oc of tile n, whose
        // copy the QK issuer has waited for (the wait here returns at once and
        // orders this thread's reads after the copy).
        if (lane == 0) {
          ok = mbar_wait(&p_full[pb], (n / PB) & 1, P.wait_limit);
          tc_fence_after();
          for (int oc = 0; oc < VS && ok; ++oc, ++consumed) {
            const int seq = SH ? n * KS + oc : consumed;
            const int ring_slots = SH ? kKSlots : kVSlots;
            const int slot = seq % ring_slots;
            if (!mbar_wait(SH ? &kfull[slot] : &vfull[slot], (seq / ring_slots) & 1, P.wait_limit)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a = smem_desc(ring_addr + slot * kTcSlotBytes, kTcHalfBytes, 1024);
            const uint64_t b = smem_desc(p_addr + pb * (kTcTok * 128), kTcHalfBytes, 1024);
#pragma unroll
            for (int k = 0; k < kTcTok / 16; ++k)  // +2048 bytes a k-step: +128 in the address field
              tc_mma(tmem_o + oc * 64, a + 128 * k, b + 128 * k, kIdescPV, (n | k) != 0);
            if (!SH) tc_commit(&vempty[slot]);
          }
          if (ok && SH)  // every K slot of tile n (the last one too) is free once its PV is done
            for (int sl = 0; sl < KS; ++sl) tc_commit(&kempty[(n * KS + sl) % kKSlots]);
          if (ok) tc_commit(&pv_done[pb]);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        consumed = __shfl_sync(0xffffffffu, consumed, 0);
        continue;
      }
      if (!warp_wait(&p_full[pb], (n / PB) & 1, lane, P.wait_limit)) { ok = false; break; }
      tc_fence_after();
      for (int oc = 0; oc < VS; ++oc, ++consumed) {
        // shared KV: chunk oc is K slot oc of tile n (already waited on by the
        // QK issuer; this wait returns at once and orders the reads after the copy)
        const int ring_slots = SH ? kKSlots : kVSlots;
        const int seq = SH ? n * KS + oc : consumed;
        const int slot = seq % ring_slots;
        if (!warp_wait(SH ? &kfull[slot] : &vfull[slot], (seq / ring_slots) & 1, lane, P.wait_limit)) { ok = false; break; }
        if (nvalid < kTcTok) {
          // V rows of tokens past the range may hold anything (NaN included):
          // zero them (both 64-dim halves) so that p = 0 contributes nothing.
          const int per = (kTcTok - nvalid) * 8;
          for (int idx = lane; idx < 2 * per; idx += 32) {
            const int h = idx / per, rem = idx % per;
            *reinterpret_cast<uint4*>(ring + slot * kTcSlotBytes + h * kTcHalfBytes +
                                      (nvalid + rem / 8) * 128 + (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < kTcTok / 16; ++k) {
            const uint64_t a = smem_desc(ring_addr + slot * kTcSlotBytes + k * 2048, kTcHalfBytes, 1024);
            const uint64_t b = smem_desc(p_addr + pb * (kTcTok * 128) + k * 2048, kTcHalfBytes, 1024);
            tc_mma(tmem_o + oc * 64, a, b, kIdescPV, (n | k) != 0);
          }
          if (!SH) tc_commit(&vempty[slot]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (SH && lane == 0)  // every K slot of tile n (the last one too) is free once its PV is done
        for (int sl = 0; sl < KS; ++sl) tc_commit(&kempty[(n * KS + sl) % kKSlots]);
      if (lane == 0) tc_commit(&pv_done[pb]);
      __syncwarp();
    }
    if (!ok && lane == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    if (lane == 0) tc_commit(o_done);  // completes when every PV MMA above is done
    __syncwarp();
  } else {
    // ================= softmax warps 2-9 =================
    // Query tile first (the producers are already streaming K and V): row r
    // of the tile, chunk c (8 dims) -> box c/8, swizzled position, in two
    // rounds whose loads are all issued before their stores. With the query
    // by TMA (P.q_tma) the producer fetches rows 0..G-1 and these warps only
    // zero the rows past them.
    {
      const int st = tid - 64;  // 0..255
      if (P.q_tma) {
        const int G = P.group;
        const int pad = (NR - G) * 8;  // 16-byte chunks per 64-dim block past row G
        for (int i = st; i < (HK / 64) * pad; i += 256)
          *reinterpret_cast<uint4*>(q_s + (i / pad) * (NR * 128) + G * 128 + (i % pad) * 16) =
              make_uint4(0, 0, 0, 0);
      } else {
        constexpr int kChunks = NR * (HK / 8);
        constexpr int kPer = (kChunks + 255) / 256;
        constexpr int kHalf = (kPer + 1) / 2;
#pragma unroll
        for (int round = 0; round < 2; ++round) {
          uint4 v[kHalf];
#pragma unroll
          for (int k = 0; k < kHalf; ++k) {
            const int idx = st + (round * kHalf + k) * 256;
            const int r = idx / (HK / 8), c = idx % (HK / 8);
            v[k] = make_uint4(0, 0, 0, 0);
            if (round * kHalf + k < kPer && idx < kChunks && r < it.nrows) {
              const int rr = it.r0 + r;
              v[k] = *reinterpret_cast<const uint4*>(
                  P.query + (int64_t(it.q_start + rr / G) * P.num_heads + it.kvh * G + rr % G) * HK + c * 8);
            }
          }
#pragma unroll
          for (int k = 0; k < kHalf; ++k) {
            const int idx = st + (round * kHalf + k) * 256;
            const int r = idx / (HK / 8), c = idx % (HK / 8);
            if (round * kHalf + k < kPer && idx < kChunks)
              *reinterpret_cast<uint4*>(q_s + (c >> 3) * (NR * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v[k];
          }
        }
      }
      if (NR < kTcRows)  // P^T columns past NR are read by the PV MMA: keep them zero
        for (int i = st; i < PB * kTcTok * 8; i += 256)
          reinterpret_cast<uint4*>(p_s)[i] = make_uint4(0, 0, 0, 0);
      fence_proxy_async();  // written by threads, read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
    }
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int rh = (warp - 2) >> 2;           // which 32 of the 64 rows
    const bool active = lane < 16;            // M=64: lanes 0-15 of a quarter hold tokens
    const int tt = quarter * 16 + lane;       // token within the tile (active lanes)
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const int rbase = rh * RH;
    // This token's probabilities summed over the tiles, for rows rbase + r,
    // relative to the row's reference max; reduced across tokens at the end.
    float l_t[RH];
#pragma unroll
    for (int r = 0; r < RH; ++r) l_t[r] = 0.f;
    const float4* m_used4 = reinterpret_cast<const float4*>(m_used + rbase);
    bool ok = true;
    for (int n = 0; n < ntiles; ++n) {
      const bool got = mbar_wait(&s_full[n & 1], (n >> 1) & 1, P.wait_limit);
      if (softmax_bar_or(!got)) { ok = false; break; }  // all softmax warps agree
      tc_fence_after();
      float s[RH];
      tmem_ld<RH>(tmem_s + (n & 1) * 64 + lane_base + rbase, s);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[n & 1]);  // this S^T buffer may be rewritten
      const int j = it.tok0 + n * kTcTok + tt;
      const bool tok_ok = active && j < it.tok1;
      // scores in base 2, plus bias; tokens past the range drop out
      if (P.mask_type == PA_MASK_ALIBI) {
#pragma unroll
        for (int r = 0; r < RH; ++r)
          s[r] = s[r] * P.scale_log2 + slope2[rbase + r] * float(j - prow[rbase + r]);
      } else {
#pragma unroll
        for (int r = 0; r < RH; ++r) s[r] *= P.scale_log2;
        // the mask is read only above the diagonal (j > p): on and below it
        // the pages fix it at 0; rows grow in position, so a token at or
        // before this warp's first row position needs no read at all
        if (P.mask_type == PA_MASK_NORM_COMPRESS && tok_ok && j > prefix + (it.r0 + rbase) / G) {
          const int mc = min(max(j - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
#pragma unroll
          for (int r = 0; r < RH; ++r) {
            const int pr = prow[rbase + r];
            if (j > pr) {
              const int mr = min(max(pr - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
              s[r] += __half2float(P.mask[mr * PA_COMPRESS_MASK_SIZE + mc]) * kLog2e;
            }
          }
        } else if (P.mask_type == PA_MASK_NORM && tok_ok) {
#pragma unroll
          for (int r = 0; r < RH; ++r) s[r] += norm_mask_log2(P, it.b, prow[rbase + r] - prefix, j);
        }
      }
      if (!tok_ok) {
#pragma unroll
        for (int r = 0; r < RH; ++r) s[r] = -INFINITY;
      }
      // Is any score above its row's reference max by more than the threshold?
      // (Always on the first tile, where the references are -inf.)
      float ex = -INFINITY;
#pragma unroll
      for (int r4 = 0; r4 < RH / 4; ++r4) {
        const float4 m = m_used4[r4];
        ex = fmaxf(ex, fmaxf(fmaxf(s[4 * r4] - m.x, s[4 * r4 + 1] - m.y),
                             fmaxf(s[4 * r4 + 2] - m.z, s[4 * r4 + 3] - m.w)));
      }
      bool grew = false;
      if (softmax_bar_or(ex > kTcRescaleThreshold)) {
        // exact tile max per row: warp max, then across the 4 lane quarters
        float keep = 0.f;
#pragma unroll
        for (int r = 0; r < RH; ++r) {
          const float wm = warp_max(s[r]);
          if (r == lane) keep = wm;
        }
        if (lane < RH) red[quarter * 64 + rbase + lane] = keep;
        softmax_bar();
        if (warp == 2) {
          bool grow = false;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int r = lane + 32 * e;
            if (r >= NR) break;
            const float mt = fmaxf(fmaxf(red[r], red[64 + r]), fmaxf(red[128 + r], red[192 + r]));
            const float mu = m_used[r];
            const float nm = fmaxf(mt, mu);
            alpha_s[r] = ex2(mu - nm);  // 0 on the first tile
            m_used[r] = nm;
            grow = grow || (mu != -INFINITY && nm != mu);
          }
          grow = __any_sync(0xffffffffu, grow);
          if (lane == 0) flags[1] = grow ? 1 : 0;
        }
        softmax_bar();
        grew = flags[1] != 0;
        if (grew) {
#pragma unroll
          for (int r = 0; r < RH; ++r) l_t[r] *= alpha_s[rbase + r];
        }
      }
      // probabilities and per-token sums
#pragma unroll
      for (int r4 = 0; r4 < RH / 4; ++r4) {
        const float4 m = m_used4[r4];
        s[4 * r4] = ex2(s[4 * r4] - m.x);
        s[4 * r4 + 1] = ex2(s[4 * r4 + 1] - m.y);
        s[4 * r4 + 2] = ex2(s[4 * r4 + 2] - m.z);
        s[4 * r4 + 3] = ex2(s[4 * r4 + 3] - m.w);
      }
#pragma unroll
      for (int r = 0; r < RH; ++r) l_t[r] += s[r];
      // P^T buffer n % PB was last read by PV(n - PB); a rescale
      // of O^T also needs PV(n - 1). Each wait is on the barrier of that PV's
      // P^T buffer, whose next phase needs P^T(n) and so cannot have begun.
      {
        bool pv = true;
        if (grew && n >= 1)
          pv = mbar_wait(&pv_done[(n - 1) % PB], ((n - 1) / PB) & 1, P.wait_limit);
        if (n >= PB)
          pv = pv && mbar_wait(&pv_done[n % PB], ((n - PB) / PB) & 1, P.wait_limit);
        if (softmax_bar_or(!pv)) { ok = false; break; }
        tc_fence_after();
      }
      // P^T into shared memory: token row tt, rows rbase.. = 16-byte chunks
      // 4 rh .. 4 rh + 3 of the 128-byte row
      if (active) {
#pragma unroll
        for (int c8 = 0; c8 < RH / 8; ++c8) {
          uint4 pk;
          pk.x = pack_half2(s[c8 * 8 + 0], s[c8 * 8 + 1]);
          pk.y = pack_half2(s[c8 * 8 + 2], s[c8 * 8 + 3]);
          pk.z = pack_half2(s[c8 * 8 + 4], s[c8 * 8 + 5]);
          pk.w = pack_half2(s[c8 * 8 + 6], s[c8 * 8 + 7]);
          const int chunk = rh * (RH / 8) + c8;
          *reinterpret_cast<uint4*>(p_s + (n % PB) * (kTcTok * 128) + tt * 128 + ((chunk ^ (tt & 7)) << 4)) = pk;
        }
      }
      if (grew) {
        // References grew: rescale this thread's O^T lane (an output dim) for
        // its 32 rows, before this tile's PV (PV of the previous tile is done).
#pragma unroll 1
        for (int oc = 0; oc < VS; ++oc) {
          float o[RH];
          const uint32_t ta = tmem_o + oc * 64 + rbase + lane_base;
          tmem_ld<RH>(ta, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < RH; ++i) o[i] *= alpha_s[rbase + i];
          tmem_st<RH>(ta, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async();  // P^T is read by the tensor cores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[n % PB]);
    }
    const int t = quarter * 32 + lane;  // TMEM lane of this thread = output dim in a chunk
    if (!ok && t == 0 && rh == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    // ---- epilogue: row sums across all tokens, then O^T / l
    {
      float mine = 0.f;  // lane l < RH: row rbase + l, summed over this warp's tokens
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        const float t = warp_sum(l_t[r]);
        if (r == lane) mine = t;
      }
      if (lane < RH) red[quarter * 64 + rbase + lane] = mine;
    }
    softmax_bar();
    const bool partial = it.slot >= 0;
    const bool fits = !partial || int64_t(it.slot) + it.nrows <= P.part_rows_cap;
    // Per-row work of the epilogue, once (warp 2): the row's 1/l, its LSE (split
    // items) and its output row (whole items). The arrays reused here are no
    // longer read by the softmax loop. Keeping this out of the per-element loop
    // keeps that loop small; a per-element version spent ~20 us per item.
    float* inv_l = alpha_s;
    int* out_row = prow;
    if (warp == 2) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = lane + 32 * e;
        if (r >= NR) break;
        const float l = (red[r] + red[64 + r]) + (red[128 + r] + red[192 + r]);
        l_tot[r] = l;
        inv_l[r] = 1.f / l;
        const int rr = it.r0 + r;
        out_row[r] = (it.q_start + rr / G) * P.num_heads + it.kvh * G + rr % G;
        if (partial && fits && r < it.nrows && ntiles > 0)
          P.part_lse[it.slot + r] = (m_used[r] + log2f(l)) * kLn2;
      }
    }
    launch_dependents();
    const bool got = ok && mbar_wait(o_done, 0, P.wait_limit);
    const bool done = !softmax_bar_or(!got);
    if (done && ntiles > 0) {
      tc_fence_after();
      if (!fits && t == 0 && rh == 0) set_status(P.status, PA_STATUS_BIT_WORKSPACE);
#pragma unroll 1
      for (int oc = 0; oc < VS; ++oc) {
        const int d = oc * 128 + t;  // output dim of this thread
        float o[RH];
        tmem_ld<RH>(tmem_o + oc * 64 + rbase + lane_base, o);
        tmem_wait_ld();
        if (!fits) continue;
        if (partial) {
          // Lanes 2k and 2k + 1 hold dims d and d + 1: each stores both (one
          // half2) for half of the 32 rows, the even lane rows rbase + i, the
          // odd lane rows rbase + RH/2 + i, taking the partner's value by
          // shuffle (128 bytes a warp store, as many bytes as an fp32 row)
          const bool odd = lane & 1;
          __half2* dst = reinterpret_cast<__half2*>(
              P.part_o + (int64_t(it.slot) + rbase + (odd ? RH / 2 : 0)) * HV + (d & ~1));
#pragma unroll
          for (int i = 0; i < RH / 2; ++i) {
            const float lo = o[i] * inv_l[rbase + i];
            const float hi = o[RH / 2 + i] * inv_l[rbase + RH / 2 + i];
            const float got = __shfl_xor_sync(0xffffffffu, odd ? lo : hi, 1);
            const float keep = odd ? hi : lo;
            const int row = rbase + (odd ? RH / 2 : 0) + i;
            if (row < it.nrows)
              dst[int64_t(i) * (HV / 2)] = odd ? __floats2half2_rn(got, keep) : __floats2half2_rn(keep, got);
          }
        } else {
#pragma unroll
          for (int i = 0; i < RH; ++i)
            if (rbase + i < it.nrows)
              P.out[int64_t(out_row[rbase + i]) * HV + d] = __float2half_rn(o[i] * inv_l[rbase + i]);
        }
      }
    } else if (done && it.slot >= 0 && int64_t(it.slot) + it.nrows <= P.part_rows_cap) {
      // an empty split (causal trim): weight zero in the combine
      for (int idx = t + 128 * rh; idx < it.nrows * HV; idx += 256) {
        P.part_o[int64_t(it.slot) * HV + idx] = __float2half_rn(0.f);
        if (idx % HV == 0) P.part_lse[it.slot + idx / HV] = -INFINITY;
      }
    }
  }
  // ---- teardown: every tcgen05 op has completed (o_done) before TMEM is freed
  // (these two waits take the default limit whatever P.wait_limit is)
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

// Launch with NR rows per tile (instantiated in pa_decode_tc.cu, _n16.cu, _n32.cu).
template <int NR>
cudaError_t launch_tc_rows(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                           const FwdParams& P, int64_t n_items, cudaStream_t stream);

// Rows per tile of a launch: the group's rows G * max_q rounded up to 16, 32 or 64.
inline int tc_tile_rows(int group, int max_q) {
  const int r = group * max_q;
  return r <= 16 ? 16 : (r <= 32 ? 32 : 64);
}

// tmq: the query as the tiles' TMA source when P.q_tma is set (one query
// token per sequence), else unused.
cudaError_t launch_tc(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                      const FwdParams& P, int64_t n_items, cudaStream_t stream);

// One launcher body for every NR: the head-size pairs of tc_supported.
template <int NR>
cudaError_t launch_tc_rows_impl(const CUtensorMap& tmk, const CUtensorMap& tmv,
                                const CUtensorMap& tmq, const FwdParams& P, int64_t n_items,
                                cudaStream_t stream,
                                cudaError_t (*set_attr)(const void*, int)) {
  auto go = [&](auto kern, uint32_t bytes) -> cudaError_t {
    cudaError_t e = set_attr(reinterpret_cast<const void*>(kern), int(bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(n_items), kTcThreads, bytes, stream>>>(tmk, tmv, tmq, P);
    return cudaGetLastError();
  };
  const bool sh = P.kv_shared != 0;
  switch (P.hk * 1000 + P.hv) {
    case 128128:
      return sh ? go(tc_decode_kernel<128, 128, NR, true>, TcCfg<128, NR, true>::bytes)
                : go(tc_decode_kernel<128, 128, NR, false>, TcCfg<128, NR>::bytes);
    case 256256:
      return sh ? go(tc_decode_kernel<256, 256, NR, true>, TcCfg<256, NR, true>::bytes)
                : go(tc_decode_kernel<256, 256, NR, false>, TcCfg<256, NR>::bytes);
    case 512512:
      return sh ? go(tc_decode_kernel<512, 512, NR, true>, TcCfg<512, NR, true>::bytes)
                : go(tc_decode_kernel<512, 512, NR, false>, TcCfg<512, NR>::bytes);
    case 576512:
      return sh ? go(tc_decode_kernel<576, 512, NR, true>, TcCfg<576, NR, true>::bytes)
                : go(tc_decode_kernel<576, 512, NR, false>, TcCfg<576, NR>::bytes);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
