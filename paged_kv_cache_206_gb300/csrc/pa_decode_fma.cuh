// Split-KV paged decode on CUDA cores, for row tiles of up to 8 rows whose
// contraction is too thin for the tensor cores (single-row tiles, and head
// sizes the mma.sync kernel is not built for). The path of the
// PagedAttentionOperation incremental phase; the split/merge structure follows
// SparseAttnSharedkvMetadata (one task per CTA, split results merged later).
//
// Per 16-token sub-tile and warp (pipeline: pa_warp_pipe.cuh):
//   QK  lane (t, half) owns token t and half of the head dims; K comes from the
//       swizzled TMA tile (conflict-free 16-byte reads), the scaled query rows
//       are fp32 broadcasts from shared memory, products accumulate in packed
//       fp32 (FFMA2); one shuffle joins the halves.
//   softmax  running max and sum in base 2 (scores carry scale * log2 e),
//       ex2.approx for the exponentials.
//   PV  lanes own 8-dim chunks of V, token groups split the 16 tokens, the
//       probabilities are broadcast from shared memory.
#pragma once

#include "pa_warp_pipe.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kFmaBufs = 2;  // pipeline depth per warp

// Kernel-specific front area: scaled query rows [rt][hk] fp32, then per-warp
// probabilities [16][2 rt] fp32.
__host__ __device__ inline uint32_t fma_front(int rt, int nw, int hk) {
  return ((uint32_t(rt) * hk * 4 + 15) / 16 * 16) + uint32_t(nw) * kSubTokens * 2 * rt * 4;
}

__host__ __device__ inline int fma_warps(int hk, int hv) { return hk + hv <= 512 ? 4 : 2; }

template <int RT, int VC, int KBW, int VBW>
__global__ void __launch_bounds__(128) fma_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                         const __grid_constant__ CUtensorMap tmv,
                                                         const FwdParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, NW = blockDim.x >> 5;
  constexpr unsigned FULL = 0xffffffffu;

  if (P.counts && int(blockIdx.x) >= P.counts[0]) return;  // past a device plan's items
  Item it;
  it.load(P, blockIdx.x);
  const int hk = P.hk, hv = P.hv, G = P.group;
  const PipeLayout lay = pipe_layout(NW, kFmaBufs, hk, hv, fma_front(RT, NW, hk), RT);
  float* q_s = reinterpret_cast<float*>(smem + 128);
  float* p_s = reinterpret_cast<float*>(smem + 128 + (uint32_t(RT) * hk * 4 + 15) / 16 * 16) +
               warp * (kSubTokens * 2 * RT);

  WarpPipe<KBW, VBW, kFmaBufs> pipe;
  pipe.init(smem, lay, P, it, &tmk, &tmv);
  const int nmine = it.nsub > warp ? (it.nsub - warp + NW - 1) / NW : 0;
  for (int n = 0; n < kFmaBufs && n < nmine; ++n) pipe.issue(n);

  // Query rows of the tile, scaled by scale * log2(e), into shared memory.
  for (int c = threadIdx.x; c < RT * (hk / 8); c += blockDim.x) {
    const int rr = c / (hk / 8), d0 = (c % (hk / 8)) * 8;
    float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (rr < it.nrows) {
      const int r = it.r0 + rr, i = r / G, h = it.kvh * G + r % G;
      const uint4 raw = *reinterpret_cast<const uint4*>(
          P.query + (int64_t(it.q_start + i) * P.num_heads + h) * hk + d0);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = h2f2(w[e]);
        v[2 * e] = f.x * P.scale_log2;
        v[2 * e + 1] = f.y * P.scale_log2;
      }
    }
    float4* dst = reinterpret_cast<float4*>(q_s + rr * hk + d0);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }

  // Per-row constants: position p of the row's query token, bias slope.
  const int prefix = it.L - it.qlen;
  const int sigma = it.L > PA_COMPRESS_MASK_SIZE ? it.L - PA_COMPRESS_MASK_SIZE : 0;
  int prow[RT];
  float slope2[RT];
#pragma unroll
  for (int rr = 0; rr < RT; ++rr) {
    const int r = it.r0 + rr;
    const bool ok = rr < it.nrows;
    prow[rr] = ok ? prefix + r / G : it.L - 1;
    slope2[rr] = (ok && P.mask_type == PA_MASK_ALIBI)
                     ? P.alibi_slopes[it.kvh * G + r % G] * kLog2e : 0.f;
  }
  __syncthreads();

  // Lane roles. 16-byte chunks per box row, and the swizzle of a box row:
  // chunk c of row t sits at c ^ ((t >> SH) & MASK) (128-byte swizzle for
  // 64-element boxes, 32-byte swizzle for 16-element boxes).
  const int t = lane & 15, half = lane >> 4;
  constexpr int kcpb = KBW / 8, vcpb = VBW / 8;
  constexpr int klg = kcpb == 8 ? 3 : 1, vlg = vcpb == 8 ? 3 : 1;
  constexpr int ksh = kcpb == 8 ? 0 : 2, vsh = vcpb == 8 ? 0 : 2;
  constexpr int kmask = kcpb == 8 ? 7 : 1, vmask = vcpb == 8 ? 7 : 1;
  constexpr uint32_t kbox_bytes = WarpPipe<KBW, VBW, kFmaBufs>::kBoxBytes;
  constexpr uint32_t vbox_bytes = WarpPipe<KBW, VBW, kFmaBufs>::vBoxBytes;
  const int kxor = (t >> ksh) & kmask;
  const int nkc = hk / 16;  // K chunks per half
  const int vchunks = hv / 8;
  // lanes per token: the smallest power of two that covers the V chunks (at
  // most 32; beyond 32 chunks a lane takes chunks cl, cl + 32, ...)
  const int lpt = vchunks > 16 ? 32 : (vchunks > 8 ? 16 : (vchunks > 4 ? 8 : (vchunks > 2 ? 4 : 2)));
  const int ng = 32 / lpt, grp = lane / lpt, cl = lane % lpt;

  float m_run[RT], l_run[RT];
  float2 o[VC][RT][4];
#pragma unroll
  for (int rr = 0; rr < RT; ++rr) {
    m_run[rr] = -INFINITY;
    l_run[rr] = 0.f;
#pragma unroll
    for (int v = 0; v < VC; ++v)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[v][rr][e] = make_float2(0.f, 0.f);
  }

  for (int n = 0; n < nmine; ++n) {
    if (!pipe.wait(n)) {
      pipe.drain(n, nmine);
      break;
    }
    const uint8_t* kb = pipe.kbuf(n);
    const uint8_t* vb = pipe.vbuf(n);
    const int tstart = it.tok0 + pipe.sub(n) * kSubTokens;
    const int nvalid = min(kSubTokens, it.tok1 - tstart);

    // ---- QK: partial dot products over this lane's half of the dims.
    float2 acc[RT], acc2[RT];
#pragma unroll
    for (int rr = 0; rr < RT; ++rr) acc[rr] = acc2[rr] = make_float2(0.f, 0.f);
    const uint8_t* krow = kb + t * (KBW * 2);
    const float* qh = q_s + half * nkc * 8;
#pragma unroll 4
    for (int k = 0; k < nkc; ++k) {
      const int cg = half * nkc + k;
      const int box = cg >> klg, cc = cg & (kcpb - 1);
      const uint4 kv = *reinterpret_cast<const uint4*>(krow + box * kbox_bytes + ((cc ^ kxor) << 4));
      const float2 k0 = h2f2(kv.x), k1 = h2f2(kv.y), k2 = h2f2(kv.z), k3 = h2f2(kv.w);
#pragma unroll
      for (int rr = 0; rr < RT; ++rr) {
        const float4* qp = reinterpret_cast<const float4*>(qh + rr * hk + k * 8);
        const float4 qa = qp[0], qb = qp[1];
        acc[rr] = fma2(make_float2(qa.x, qa.y), k0, acc[rr]);
        acc2[rr] = fma2(make_float2(qa.z, qa.w), k1, acc2[rr]);
        acc[rr] = fma2(make_float2(qb.x, qb.y), k2, acc[rr]);
        acc2[rr] = fma2(make_float2(qb.z, qb.w), k3, acc2[rr]);
      }
    }

    // ---- scores, bias, tile max, online softmax update
    const int j = tstart + t;
    const bool tok_ok = t < nvalid;
    float s[RT], alpha[RT];
    bool rescale = false;
#pragma unroll
    for (int rr = 0; rr < RT; ++rr) {
      float x = (acc[rr].x + acc2[rr].x) + (acc[rr].y + acc2[rr].y);
      x += __shfl_xor_sync(FULL, x, 16);
      if (P.mask_type == PA_MASK_ALIBI) {
        x += slope2[rr] * float(j - prow[rr]);
      } else if (P.mask_type == PA_MASK_NORM_COMPRESS) {
        if (tok_ok && j > prow[rr]) {  // above the diagonal only
          // both indices lie in [0, 2048) for a consistent plan; clamp anyway
          const int mr = min(max(prow[rr] - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
          const int mc = min(max(j - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
          x += __half2float(P.mask[mr * PA_COMPRESS_MASK_SIZE + mc]) * kLog2e;
        }
      } else if (P.mask_type == PA_MASK_NORM) {
        if (tok_ok) x += norm_mask_log2(P, it.b, prow[rr] - prefix, j);
      }
      x = tok_ok ? x : -INFINITY;
      float mt = x;
      mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 2));
      mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 4));
      mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 8));
      const float mn = fmaxf(m_run[rr], mt);
      alpha[rr] = ex2(m_run[rr] - mn);
      rescale |= (mn != m_run[rr]);
      m_run[rr] = mn;
      s[rr] = ex2(x - mn);
      l_run[rr] = l_run[rr] * alpha[rr] + s[rr];
    }
    if (half == 0) {
      float2* pw = reinterpret_cast<float2*>(p_s + t * 2 * RT);
#pragma unroll
      for (int rr = 0; rr < RT; ++rr) pw[rr] = make_float2(s[rr], s[rr]);
    }
    if (rescale) {
#pragma unroll
      for (int rr = 0; rr < RT; ++rr) {
        const float2 a2 = make_float2(alpha[rr], alpha[rr]);
#pragma unroll
        for (int v = 0; v < VC; ++v)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[v][rr][e] = mul2(o[v][rr][e], a2);
      }
    }
    __syncwarp();

    // ---- PV: this lane's V chunks for its token group.
    for (int tt = grp; tt < nvalid; tt += ng) {
      float2 pp[RT];
      if constexpr (RT == 1) {
        pp[0] = *reinterpret_cast<const float2*>(p_s + tt * 2);
      } else {
        const float4* pr = reinterpret_cast<const float4*>(p_s + tt * 2 * RT);
#pragma unroll
        for (int h2 = 0; h2 < RT / 2; ++h2) {
          const float4 x = pr[h2];
          pp[2 * h2] = make_float2(x.x, x.y);
          pp[2 * h2 + 1] = make_float2(x.z, x.w);
        }
      }
      const int vxor = (tt >> vsh) & vmask;
      const uint8_t* vrow = vb + tt * (VBW * 2);
#pragma unroll
      for (int v = 0; v < VC; ++v) {
        const int cg = cl + 32 * v;
        if (cl < vchunks && cg < vchunks) {
          const int box = cg >> vlg, cc = cg & (vcpb - 1);
          const uint4 vv = *reinterpret_cast<const uint4*>(vrow + box * vbox_bytes + ((cc ^ vxor) << 4));
          const float2 v0 = h2f2(vv.x), v1 = h2f2(vv.y), v2 = h2f2(vv.z), v3 = h2f2(vv.w);
#pragma unroll
          for (int rr = 0; rr < RT; ++rr) {
            o[v][rr][0] = fma2(pp[rr], v0, o[v][rr][0]);
            o[v][rr][1] = fma2(pp[rr], v1, o[v][rr][1]);
            o[v][rr][2] = fma2(pp[rr], v2, o[v][rr][2]);
            o[v][rr][3] = fma2(pp[rr], v3, o[v][rr][3]);
          }
        }
      }
    }
    pipe.release_and_refill(n, nmine);
  }

  launch_dependents();  // the combine pass may be scheduled now

  // ---- warp-level reduction of the softmax sums and of the token groups.
#pragma unroll
  for (int rr = 0; rr < RT; ++rr) {
    float l = l_run[rr];
    l += __shfl_xor_sync(FULL, l, 1);
    l += __shfl_xor_sync(FULL, l, 2);
    l += __shfl_xor_sync(FULL, l, 4);
    l += __shfl_xor_sync(FULL, l, 8);
    l_run[rr] = l;
  }
  for (int off = lpt; off < 32; off <<= 1) {
#pragma unroll
    for (int v = 0; v < VC; ++v)
#pragma unroll
      for (int rr = 0; rr < RT; ++rr)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[v][rr][e].x += __shfl_xor_sync(FULL, o[v][rr][e].x, off);
          o[v][rr][e].y += __shfl_xor_sync(FULL, o[v][rr][e].y, off);
        }
  }
  __syncthreads();  // every warp is done with its buffers

  // ---- per-warp state into shared memory: m[RT], l[RT], O[RT][hv]
  float* merge = reinterpret_cast<float*>(smem + lay.buf_off);
  float* mg = merge + warp * merge_stride(RT, hv);
  if (lane == 0) {
#pragma unroll
    for (int rr = 0; rr < RT; ++rr) {
      mg[rr] = m_run[rr];
      mg[RT + rr] = l_run[rr];
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int v = 0; v < VC; ++v) {
      const int cg = cl + 32 * v;
      if (cl < vchunks && cg < vchunks) {
#pragma unroll
        for (int rr = 0; rr < RT; ++rr) {
          float4* dst = reinterpret_cast<float4*>(mg + merge_opart(RT) + rr * hv + cg * 8);
          dst[0] = make_float4(o[v][rr][0].x, o[v][rr][0].y, o[v][rr][1].x, o[v][rr][1].y);
          dst[1] = make_float4(o[v][rr][2].x, o[v][rr][2].y, o[v][rr][3].x, o[v][rr][3].y);
        }
      }
    }
  }
  __syncthreads();
  merge_store<RT>(P, it, merge, NW);
}

// Host launcher for one row-tile height; the value head size picks the
// chunks-per-lane instantiation, the head sizes pick the TMA box width.
template <int RT>
cudaError_t launch_fma(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                       int64_t n_items, cudaStream_t stream) {
  const int nw = fma_warps(P.hk, P.hv);
  const PipeLayout lay = pipe_layout(nw, kFmaBufs, P.hk, P.hv, fma_front(RT, nw, P.hk), RT);
  const int vc = (P.hv / 8 + 31) / 32;
  const bool wide = (P.hk % 64 == 0) && (P.hv % 64 == 0);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), int(lay.bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(n_items), nw * 32, lay.bytes, stream>>>(tmk, tmv, P);
    return cudaGetLastError();
  };
  if (wide) {
    switch (vc) {
      case 1: return go(fma_decode_kernel<RT, 1, 64, 64>);
      case 2: return go(fma_decode_kernel<RT, 2, 64, 64>);
      default: return go(fma_decode_kernel<RT, 3, 64, 64>);
    }
  }
  switch (vc) {
    case 1: return go(fma_decode_kernel<RT, 1, 16, 16>);
    case 2: return go(fma_decode_kernel<RT, 2, 16, 16>);
    default: return go(fma_decode_kernel<RT, 3, 16, 16>);
  }
}

}  // namespace pa
