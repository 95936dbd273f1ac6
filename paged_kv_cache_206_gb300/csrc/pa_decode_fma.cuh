// Split-KV paged decode on CUDA cores, for query-row tiles of at most 8 rows
// (one new token per sequence, or a few speculative tokens, times a small GQA
// group). This is the path of the PagedAttentionOperation incremental phase;
// the split/merge structure follows SparseAttnSharedkvMetadata (one task per
// CTA, split results merged by a later reduction).
//
// One CTA runs one work item: a (sequence, kv head, row tile, KV-block range).
// Each warp owns every NW-th 16-token sub-tile of the range and runs its own
// two-deep TMA pipeline into its own shared-memory buffers, so the main loop
// has no CTA-wide barrier; warps merge their softmax states at the end.
//
// Per sub-tile and warp:
//   QK  lane (t, half) owns token t and half of the head dims; K is read from
//       a TMA-swizzled tile (conflict-free 16-byte reads), the scaled query
//       rows are fp32 broadcasts from shared memory, products accumulate in
//       packed fp32 (fma.rn.f32x2); one shuffle joins the halves.
//   softmax  running max and sum in base 2 (scores carry scale * log2 e),
//       ex2.approx for the exponentials.
//   PV  lanes own 8-dim chunks of V, token groups split the 16 tokens, the
//       probabilities are broadcast from shared memory.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kFmaTokens = 16;  // tokens per sub-tile (one TMA box height)
constexpr int kFmaBufs = 2;     // pipeline depth per warp

// Floats per warp in the merge area: m[rt], l[rt] padded to 4, then O[rt][hv].
__host__ __device__ inline uint32_t fma_merge_stride(int rt, int hv) {
  return uint32_t((2 * rt + 3) / 4 * 4 + rt * hv);
}

struct FmaLayout {
  uint32_t q_off, p_off, buf_off, buf_stride, v_in_buf, merge_off, bytes;
};

// Shared-memory layout; the same function sizes the launch on the host.
__host__ __device__ inline FmaLayout fma_layout(int rt, int nw, int hk, int hv) {
  auto up = [](uint32_t x, uint32_t a) { return (x + a - 1) / a * a; };
  FmaLayout L;
  const uint32_t bars = 128;  // nw * kFmaBufs mbarriers
  L.q_off = bars;
  L.p_off = up(L.q_off + uint32_t(rt) * hk * 4, 16);
  const uint32_t p_bytes = uint32_t(nw) * kFmaTokens * 2 * rt * 4;
  L.buf_off = up(L.p_off + p_bytes, 1024);
  const uint32_t kbytes = up(uint32_t(kFmaTokens) * hk * 2, 1024);
  L.v_in_buf = kbytes;
  L.buf_stride = up(kbytes + uint32_t(kFmaTokens) * hv * 2, 1024);
  L.merge_off = L.buf_off;  // reused after the last tile
  const uint32_t bufs_end = L.buf_off + uint32_t(nw) * kFmaBufs * L.buf_stride;
  const uint32_t merge_end = L.merge_off + uint32_t(nw) * fma_merge_stride(rt, hv) * 4;
  L.bytes = (bufs_end > merge_end ? bufs_end : merge_end) + 1024;  // + base alignment slack
  return L;
}

__host__ __device__ inline int fma_warps(int hk, int hv) { return hk + hv <= 512 ? 4 : 2; }

template <int RT, int VC>
__global__ void __launch_bounds__(128) fma_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                         const __grid_constant__ CUtensorMap tmv,
                                                         const FwdParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, NW = blockDim.x >> 5;
  constexpr unsigned FULL = 0xffffffffu;

  const int32_t* item = P.work + int64_t(blockIdx.x) * PA_WORK_INTS;
  const int b = item[0], kvh = item[1], r0 = item[2], r1 = item[3];
  const int kb0 = item[4], kb1 = item[5], q_start = item[6], slot = item[7];
  const int nrows = r1 - r0;
  const int L = P.context_lens[b];
  const int qlen = P.q_seqlens ? P.q_seqlens[b] : 1;
  const int hk = P.hk, hv = P.hv, bs = P.block_size, G = P.group;

  const FmaLayout lay = fma_layout(RT, NW, hk, hv);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + warp * kFmaBufs;
  float* q_s = reinterpret_cast<float*>(smem + lay.q_off);
  float* p_s = reinterpret_cast<float*>(smem + lay.p_off) + warp * (kFmaTokens * 2 * RT);
  uint8_t* my_bufs = smem + lay.buf_off + uint32_t(warp) * kFmaBufs * lay.buf_stride;

  // Token range of this item and this warp's share of its sub-tiles.
  const int tok0 = kb0 * bs;
  const int tok1 = min(kb1 * bs, L);
  const int U = (tok1 - tok0 + kFmaTokens - 1) / kFmaTokens;
  const int nmine = U > warp ? (U - warp + NW - 1) / NW : 0;

  if (lane == 0) {
    for (int k = 0; k < kFmaBufs; ++k) mbar_init(&bars[k], 1);
    fence_barrier_init();
  }
  __syncwarp();

  const uint64_t pol = policy_evict_first();
  // Block-table window: lane k holds the entry of block kb0 + bt_base + k.
  const int32_t* bt_row = P.block_tables + int64_t(b) * P.max_blocks_per_seq;
  int bt_base = 0;
  int bt_reg = (kb0 + lane < kb1) ? bt_row[kb0 + lane] : 0;
  const uint32_t tile_bytes = uint32_t(kFmaTokens) * (hk + hv) * 2;
  const int nkbox = hk / P.kbw, nvbox = hv / P.vbw;
  const uint32_t kbox_bytes = uint32_t(kFmaTokens) * P.kbw * 2;
  const uint32_t vbox_bytes = uint32_t(kFmaTokens) * P.vbw * 2;

  // Warp-collective: start the TMA copies of this warp's n-th sub-tile.
  auto issue = [&](int n, int buf) {
    const int u = warp + n * NW;
    const int rel = (u * kFmaTokens) / bs;
    const int off = (u * kFmaTokens) % bs;
    if (rel >= bt_base + 32) {
      bt_base = rel & ~31;
      bt_reg = (kb0 + bt_base + lane < kb1) ? bt_row[kb0 + bt_base + lane] : 0;
    }
    const int phys = __shfl_sync(FULL, bt_reg, rel - bt_base);
    if (lane == 0) {
      if (phys < 0 || phys >= P.num_blocks) {
        // Never dereference a bad entry: flag it and complete the phase
        // without a copy (the tile's scores are then meaningless, and the
        // status word says so).
        set_status(P.status, PA_STATUS_BIT_BLOCK_INDEX);
        mbar_arrive(&bars[buf]);
        return;
      }
      const int row = phys * bs + off;
      uint8_t* dst = my_bufs + buf * lay.buf_stride;
      mbar_arrive_expect_tx(&bars[buf], tile_bytes);
      for (int j = 0; j < nkbox; ++j)
        tma_load_2d(dst + j * kbox_bytes, &tmk, &bars[buf], kvh * hk + j * P.kbw, row, pol);
      for (int j = 0; j < nvbox; ++j)
        tma_load_2d(dst + lay.v_in_buf + j * vbox_bytes, &tmv, &bars[buf], kvh * hv + j * P.vbw,
                    row, pol);
    }
  };

  for (int n = 0; n < kFmaBufs && n < nmine; ++n) issue(n, n);

  // Query rows of the tile, scaled by scale * log2(e), into shared memory.
  for (int c = threadIdx.x; c < RT * (hk / 8); c += blockDim.x) {
    const int rr = c / (hk / 8), d0 = (c % (hk / 8)) * 8;
    float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (rr < nrows) {
      const int r = r0 + rr, i = r / G, h = kvh * G + r % G;
      const uint4 raw = *reinterpret_cast<const uint4*>(
          P.query + (int64_t(q_start + i) * P.num_heads + h) * hk + d0);
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
  const int prefix = L - qlen;
  const int sigma = L > PA_COMPRESS_MASK_SIZE ? L - PA_COMPRESS_MASK_SIZE : 0;
  int prow[RT];
  float slope2[RT];
#pragma unroll
  for (int rr = 0; rr < RT; ++rr) {
    const int r = r0 + rr;
    const bool ok = rr < nrows;
    prow[rr] = ok ? prefix + r / G : L - 1;
    slope2[rr] = (ok && P.mask_type == PA_MASK_ALIBI) ? P.alibi_slopes[kvh * G + r % G] * kLog2e : 0.f;
  }
  __syncthreads();

  // Lane roles.
  const int t = lane & 15, half = lane >> 4;
  const int kcpb = P.kbw / 8, vcpb = P.vbw / 8;  // 16-byte chunks per box row
  const int kxor = (t >> (kcpb == 8 ? 0 : kcpb == 4 ? 1 : 2)) & P.kswz;
  const int nkc = hk / 16;  // K chunks per half
  const int vchunks = hv / 8;
  const int lpt = vchunks >= 32 ? 32 : (vchunks > 8 ? 16 : (vchunks > 4 ? 8 : (vchunks > 2 ? 4 : 2)));
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

  int failed_at = -1;
  for (int n = 0; n < nmine; ++n) {
    const int buf = n % kFmaBufs;
    if (!mbar_wait(&bars[buf], (n / kFmaBufs) & 1)) {
      failed_at = n;
      break;
    }
    const uint8_t* kb = my_bufs + buf * lay.buf_stride;
    const uint8_t* vb = kb + lay.v_in_buf;
    const int tstart = tok0 + (warp + n * NW) * kFmaTokens;
    const int nvalid = min(kFmaTokens, tok1 - tstart);

    // ---- QK: partial dot products over this lane's half of the dims.
    float2 acc[RT];
#pragma unroll
    for (int rr = 0; rr < RT; ++rr) acc[rr] = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int k = 0; k < nkc; ++k) {
      const int cg = half * nkc + k;
      const int box = cg / kcpb, cc = cg % kcpb;
      const uint4 kv = *reinterpret_cast<const uint4*>(
          kb + box * kbox_bytes + t * (P.kbw * 2) + ((cc ^ kxor) << 4));
      const float2 k0 = h2f2(kv.x), k1 = h2f2(kv.y), k2 = h2f2(kv.z), k3 = h2f2(kv.w);
#pragma unroll
      for (int rr = 0; rr < RT; ++rr) {
        const float4* qp = reinterpret_cast<const float4*>(q_s + rr * hk + cg * 8);
        const float4 qa = qp[0], qb = qp[1];
        acc[rr] = fma2(make_float2(qa.x, qa.y), k0, acc[rr]);
        acc[rr] = fma2(make_float2(qa.z, qa.w), k1, acc[rr]);
        acc[rr] = fma2(make_float2(qb.x, qb.y), k2, acc[rr]);
        acc[rr] = fma2(make_float2(qb.z, qb.w), k3, acc[rr]);
      }
    }

    // ---- scores, bias, tile max, online softmax update
    const int j = tstart + t;
    const bool tok_ok = t < nvalid;
    float s[RT], alpha[RT];
    bool rescale = false;
#pragma unroll
    for (int rr = 0; rr < RT; ++rr) {
      float x = acc[rr].x + acc[rr].y;
      x += __shfl_xor_sync(FULL, x, 16);
      if (P.mask_type == PA_MASK_ALIBI) {
        x += slope2[rr] * float(j - prow[rr]);
      } else if (P.mask_type == PA_MASK_NORM_COMPRESS) {
        if (tok_ok && j > prefix) {
          // both indices lie in [0, 2048) for a consistent plan; clamp anyway
          const int mr = min(max(prow[rr] - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
          const int mc = min(max(j - sigma, 0), PA_COMPRESS_MASK_SIZE - 1);
          x += __half2float(P.mask[mr * PA_COMPRESS_MASK_SIZE + mc]) * kLog2e;
        }
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
      const float4* pr = reinterpret_cast<const float4*>(p_s + tt * 2 * RT);
      if constexpr (RT == 1) {
        pp[0] = *reinterpret_cast<const float2*>(p_s + tt * 2);
      } else {
#pragma unroll
        for (int h2 = 0; h2 < RT / 2; ++h2) {
          const float4 x = pr[h2];
          pp[2 * h2] = make_float2(x.x, x.y);
          pp[2 * h2 + 1] = make_float2(x.z, x.w);
        }
      }
      const int vxor = (tt >> (vcpb == 8 ? 0 : vcpb == 4 ? 1 : 2)) & P.vswz;
#pragma unroll
      for (int v = 0; v < VC; ++v) {
        const int cg = cl + 32 * v;
        if (cl < vchunks && cg < vchunks) {
          const int box = cg / vcpb, cc = cg % vcpb;
          const uint4 vv = *reinterpret_cast<const uint4*>(
              vb + box * vbox_bytes + tt * (P.vbw * 2) + ((cc ^ vxor) << 4));
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
    __syncwarp();
    fence_proxy_async();
    if (n + kFmaBufs < nmine) issue(n + kFmaBufs, buf);
  }

  if (failed_at >= 0) {
    if (lane == 0) set_status(P.status, PA_STATUS_BIT_TIMEOUT);
    // Let the copies still in flight (sub-tiles failed_at .. failed_at + depth)
    // land before this CTA's shared memory is released; each wait is bounded.
    for (int m = failed_at; m < failed_at + kFmaBufs && m < nmine; ++m)
      mbar_wait(&bars[m % kFmaBufs], (m / kFmaBufs) & 1);
  }

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
  const int mstride = int(fma_merge_stride(RT, hv));
  const int opart = (2 * RT + 3) / 4 * 4;
  float* mg = reinterpret_cast<float*>(smem + lay.merge_off) + warp * mstride;
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
          float4* dst = reinterpret_cast<float4*>(mg + opart + rr * hv + cg * 8);
          dst[0] = make_float4(o[v][rr][0].x, o[v][rr][0].y, o[v][rr][1].x, o[v][rr][1].y);
          dst[1] = make_float4(o[v][rr][2].x, o[v][rr][2].y, o[v][rr][3].x, o[v][rr][3].y);
        }
      }
    }
  }
  __syncthreads();

  // ---- merge the warps and write the output or the partial result
  const bool partial = slot >= 0;
  if (partial && int64_t(slot) + nrows > P.part_rows_cap) {
    if (threadIdx.x == 0) set_status(P.status, PA_STATUS_BIT_WORKSPACE);
    return;
  }
  const float* base = reinterpret_cast<const float*>(smem + lay.merge_off);
  for (int idx = threadIdx.x; idx < nrows * hv; idx += blockDim.x) {
    const int rr = idx / hv, d = idx % hv;
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, base[w * mstride + rr]);
    float lsum = 0.f, osum = 0.f;
    for (int w = 0; w < NW; ++w) {
      const float* ww = base + w * mstride;
      const float f = ex2(ww[rr] - M);
      lsum += ww[RT + rr] * f;
      osum += ww[opart + rr * hv + d] * f;
    }
    const float val = osum / lsum;
    if (!partial) {
      const int r = r0 + rr, i = r / G, h = kvh * G + r % G;
      P.out[(int64_t(q_start + i) * P.num_heads + h) * hv + d] = __float2half_rn(val);
    } else {
      P.part_o[(int64_t(slot) + rr) * hv + d] = val;
      if (d == 0) P.part_lse[slot + rr] = (M + log2f(lsum)) * kLn2;
    }
  }
}

}  // namespace pa

namespace pa {

// Host launcher for one row-tile height; the value head size picks the
// chunks-per-lane instantiation.
template <int RT>
cudaError_t launch_fma(const CUtensorMap& tmk, const CUtensorMap& tmv, const FwdParams& P,
                       int64_t n_items, cudaStream_t stream) {
  const int nw = fma_warps(P.hk, P.hv);
  const FmaLayout lay = fma_layout(RT, nw, P.hk, P.hv);
  const int vc = (P.hv / 8 + 31) / 32;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(lay.bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(n_items), nw * 32, lay.bytes, stream>>>(tmk, tmv, P);
    return cudaGetLastError();
  };
  switch (vc) {
    case 1: return go(fma_decode_kernel<RT, 1>);
    case 2: return go(fma_decode_kernel<RT, 2>);
    default: return go(fma_decode_kernel<RT, 3>);
  }
}

}  // namespace pa
