// Split-KV paged decode on the tensor cores' warp-level MMA, for row tiles of
// 2..8 rows (a GQA group times a few query tokens): the tile is a real, if
// thin, dense contraction, and the CUDA-core kernel spends most of its issue
// slots and shared-memory bandwidth on query broadcasts and fp16 conversions
// at these shapes. PagedAttentionOperation incremental phase; the split/merge
// structure follows SparseAttnSharedkvMetadata.
//
// Per 16-token sub-tile and warp (pipeline: pa_warp_pipe.cuh), with the
// operands swapped so that the 16 tokens fill the M side of m16n8k16 and the
// up-to-8 query rows the N side:
//   S^T[16 tok x 8 rows]  = K[16 x hk] . Q^T[hk x 8]   (Q^T fragments stay in
//                           registers for the whole item; K via ldmatrix from
//                           the 128-byte-swizzled TMA tile, conflict-free)
//   online softmax on S^T in base 2 (row max over the 16 tokens: one in-lane
//                           max and three shuffles)
//   P^T fragments         = movmatrix.trans of the fp16-packed S^T fragments
//   O^T[hv x 8]          += V^T[hv x 16 tok] . P^T     (V via ldmatrix.trans)
// fp32 accumulation throughout; P is rounded to fp16 for the PV product.
#pragma once

#include "pa_warp_pipe.cuh"

namespace pa {

constexpr int kMmaBufs = 2;

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// d += a . b, m16n8k16, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__host__ __device__ inline int mma_warps(int hk, int hv) { return hk + hv <= 512 ? 4 : 2; }

template <int HK, int HV>
__global__ void __launch_bounds__(128) mma_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                         const __grid_constant__ CUtensorMap tmv,
                                                         const FwdParams P) {
  constexpr int KS = HK / 16;  // k-steps of QK
  constexpr int MT = HV / 16;  // m-tiles of PV
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, NW = blockDim.x >> 5;
  const int g = lane >> 2, c = lane & 3;

  if (P.counts && int(blockIdx.x) >= P.counts[0]) return;  // past a device plan's items
  Item it;
  it.load(P, blockIdx.x);
  const int G = P.group;
  const PipeLayout lay = pipe_layout(NW, kMmaBufs, HK, HV, 0, 8);
  WarpPipe<64, 64, kMmaBufs> pipe;
  pipe.init(smem, lay, P, it, &tmk, &tmv);
  const int nmine = it.nsub > warp ? (it.nsub - warp + NW - 1) / NW : 0;
  for (int n = 0; n < kMmaBufs && n < nmine; ++n) pipe.issue(n);

  // Q^T fragments: B[k = dim][n = row] for row g of the tile.
  uint32_t qf[KS][2];
  {
    const bool ok = g < it.nrows;
    const int r = it.r0 + g;
    const __half* qrow =
        P.query + (int64_t(it.q_start + (ok ? r / G : 0)) * P.num_heads + it.kvh * G + (ok ? r % G : 0)) * HK;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qf[ks][0] = ok ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * c) : 0u;
      qf[ks][1] = ok ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * c) : 0u;
    }
  }
  // This lane's two score columns are tile rows 2c and 2c + 1.
  const int prefix = it.L - it.qlen;
  const int sigma = it.L > PA_COMPRESS_MASK_SIZE ? it.L - PA_COMPRESS_MASK_SIZE : 0;
  int prow[2];
  float slope2[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int rr = 2 * c + e, r = it.r0 + rr;
    const bool ok = rr < it.nrows;
    prow[e] = ok ? prefix + r / G : it.L - 1;
    slope2[e] = (ok && P.mask_type == PA_MASK_ALIBI)
                    ? P.alibi_slopes[it.kvh * G + r % G] * kLog2e : 0.f;
  }

  // ldmatrix row providers: QK (plain) and PV (transposed) address patterns.
  const int ta = (lane & 7) + ((lane >> 3) & 1) * 8, ca = lane >> 4;
  const int tv = (lane & 7) + (lane >> 4) * 8, cv = (lane >> 3) & 1;

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  for (int n = 0; n < nmine; ++n) {
    if (!pipe.wait(n)) {
      pipe.drain(n, nmine);
      break;
    }
    const uint8_t* kb = pipe.kbuf(n);
    uint8_t* vb = pipe.vbuf(n);
    const int tstart = it.tok0 + pipe.sub(n) * kSubTokens;
    const int nvalid = min(kSubTokens, it.tok1 - tstart);

    // ---- S^T = K . Q^T
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    const uint8_t* krow = kb + ta * 128;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int cc = ((ks & 3) << 1) + ca;
      uint32_t a[4];
      ldsm_x4(a, krow + (ks >> 2) * 2048 + ((cc ^ (ta & 7)) << 4));
      mma_16816(s, a, qf[ks][0], qf[ks][1]);
    }

    // ---- scale, bias, tail, online softmax. s[0]: (token g, row 2c),
    // s[1]: (g, 2c+1), s[2]: (g+8, 2c), s[3]: (g+8, 2c+1).
    float x[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tok = g + (e >> 1) * 8, col = e & 1;
      const int j = tstart + tok;
      float v = s[e] * P.scale_log2;
      if (P.mask_type == PA_MASK_ALIBI) {
        v += slope2[col] * float(j - prow[col]);
      } else if (P.mask_type == PA_MASK_NORM_COMPRESS) {
        if (tok < nvalid && j > prow[col]) {  // above the diagonal only
          const int mr = min(max(prow[col] - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
          const int mc = min(max(j - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
          v += __half2float(P.mask[mr * PA_COMPRESS_MASK_SIZE + mc]) * kLog2e;
        }
      } else if (P.mask_type == PA_MASK_NORM) {
        if (tok < nvalid) v += norm_mask_log2(P, it.b, prow[col] - prefix, j);
      }
      x[e] = tok < nvalid ? v : -INFINITY;
    }
    float alpha[2];
    bool rescale = false;
#pragma unroll
    for (int col = 0; col < 2; ++col) {
      float mt = fmaxf(x[col], x[col + 2]);
      mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 4));
      mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 8));
      mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 16));
      const float mn = fmaxf(m_run[col], mt);
      alpha[col] = ex2(m_run[col] - mn);
      rescale |= (mn != m_run[col]);
      m_run[col] = mn;
    }
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = ex2(x[e] - m_run[e & 1]);
    l_run[0] = l_run[0] * alpha[0] + (p[0] + p[2]);
    l_run[1] = l_run[1] * alpha[1] + (p[1] + p[3]);
    if (__any_sync(FULL, rescale)) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] *= alpha[0];
        o[mt][1] *= alpha[1];
        o[mt][2] *= alpha[0];
        o[mt][3] *= alpha[1];
      }
    }
    const uint32_t pb0 = movmatrix_t(pack_half2(p[0], p[1]));  // tokens 0-7
    const uint32_t pb1 = movmatrix_t(pack_half2(p[2], p[3]));  // tokens 8-15

    // Tokens past the context (tail of the last block) carry p = 0, but their
    // V slots may hold anything, NaN included: zero those rows first.
    if (nvalid < kSubTokens) {
      const int rows = kSubTokens - nvalid;
      for (int idx = lane; idx < rows * 8 * (HV / 64); idx += 32) {
        const int box = idx / (rows * 8), rem = idx % (rows * 8);
        const int t = nvalid + rem / 8, ch = rem % 8;
        *reinterpret_cast<uint4*>(vb + box * 2048 + t * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }

    // ---- O^T += V^T . P^T
    const uint8_t* vrow = vb + tv * 128;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int cc = ((mt & 3) << 1) + cv;
      uint32_t a[4];
      ldsm_x4_t(a, vrow + (mt >> 2) * 2048 + ((cc ^ (tv & 7)) << 4));
      mma_16816(o[mt], a, pb0, pb1);
    }
    pipe.release_and_refill(n, nmine);
  }

  launch_dependents();  // the combine pass may be scheduled now

  // ---- reduce l over the lanes that share a row pair (same c)
#pragma unroll
  for (int col = 0; col < 2; ++col) {
    float l = l_run[col];
    l += __shfl_xor_sync(FULL, l, 4);
    l += __shfl_xor_sync(FULL, l, 8);
    l += __shfl_xor_sync(FULL, l, 16);
    l_run[col] = l;
  }
  __syncthreads();  // every warp is done with its buffers

  // ---- per-warp state into shared memory: m[8], l[8], O[8][HV]
  float* merge = reinterpret_cast<float*>(smem + lay.buf_off);
  float* mg = merge + warp * merge_stride(8, HV);
  if (g == 0) {
    mg[2 * c] = m_run[0];
    mg[2 * c + 1] = m_run[1];
    mg[8 + 2 * c] = l_run[0];
    mg[8 + 2 * c + 1] = l_run[1];
  }
  float* og = mg + merge_opart(8);
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int d = mt * 16 + g;
    og[(2 * c) * HV + d] = o[mt][0];
    og[(2 * c + 1) * HV + d] = o[mt][1];
    og[(2 * c) * HV + d + 8] = o[mt][2];
    og[(2 * c + 1) * HV + d + 8] = o[mt][3];
  }
  __syncthreads();
  merge_store<8>(P, it, merge, NW);
}

// Head-size pairs the mma.sync kernel is instantiated for.
inline bool mma_supported(int hk, int hv) {
  return (hk == hv && (hk == 64 || hk == 128 || hk == 256 || hk == 512)) ||
         (hk == 576 && hv == 512);
}

cudaError_t launch_mma(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                       int64_t n_items, cudaStream_t stream);

}  // namespace pa
