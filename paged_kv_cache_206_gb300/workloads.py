"""Seeded synthetic inputs for paged attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic. Both the CUDA path and the CPU oracle consume what it
produces, so neither side's correctness can leak into the other's inputs.

Shapes follow the paged KV cache of the PagedAttentionOperation pages
("Constraints"): ``key_cache``/``value_cache`` are
``[num_blocks, block_size, kv_heads, head_size]`` fp16, ``block_tables`` is
``[batch, max_num_blocks_per_seq]`` int32 with every entry in
``[0, num_blocks)``, ``context_lens`` counts the whole KV length of a sequence
including its current query tokens, and ``max_num_blocks_per_seq`` is at least
``ceil(max(context_lens) / block_size)``. Queries use the token-concatenated
layout of the SparseAttnSharedkvMetadata page ("参数说明", ``cu_seqlens_q``):
``query[sum(q_seqlens), num_heads, head_size]``.

Determinism: every large array is drawn in fixed chunks of ``_CHUNK`` values,
chunk ``k`` from the ``k``-th child of ``SeedSequence(seed)``, so the bits do
not depend on how many threads fill them.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

MASK_NONE = 0
MASK_NORM = 1
MASK_ALIBI = 2
MASK_NORM_COMPRESS = 5

COMPRESS_MASK_SIZE = 2048
_CHUNK = 1 << 22


@dataclass
class Workload:
    """One batch of paged-attention inputs (host numpy arrays)."""

    name: str
    num_heads: int
    kv_heads: int
    head_size_k: int
    head_size_v: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    mask_type: int
    scale: float
    context_lens: np.ndarray  # int32 [B]
    q_seqlens: np.ndarray  # int32 [B]
    block_tables: np.ndarray  # int32 [B, max_blocks_per_seq]
    query: np.ndarray  # fp16 [sum q, H, hk]
    key_cache: np.ndarray  # fp16 [nb, bs, Hk, hk]
    value_cache: np.ndarray  # fp16 [nb, bs, Hk, hv]
    mask: np.ndarray | None = None  # fp16 [2048, 2048], or [B, max q, maxNB * bs] (NORM)
    alibi_slopes: np.ndarray | None = None  # fp32 [H]
    chunk_blocks: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_seqlen_q(self) -> int:
        return int(self.q_seqlens.max())

    @property
    def total_q(self) -> int:
        return int(self.q_seqlens.sum())

    @property
    def shared_kv(self) -> bool:
        return bool(self.meta.get("shared_kv", False))

    def kv_bytes(self) -> int:
        """Bytes of K and V that attention must read: sum_b L_b * Hk * (hk + hv) * 2,
        or sum_b L_b * Hk * hk * 2 when V is part of the K rows (shared cache)."""
        per = self.head_size_k + (0 if self.shared_kv else self.head_size_v)
        return int(self.context_lens.astype(np.int64).sum()) * self.kv_heads * per * 2

    def attn_flops(self) -> int:
        """Multiply-add flops of QK^T and PV over the keys each query row sees:
        2 * (hk + hv) per (row, key); with the causal mask row i of a sequence
        sees L - q + i + 1 keys, otherwise all L."""
        L = self.context_lens.astype(np.int64)
        q = self.q_seqlens.astype(np.int64)
        if self.mask_type == MASK_NORM_COMPRESS:
            pairs = (q * (L - q) + q * (q + 1) // 2).sum()
        else:
            pairs = (q * L).sum()
        return int(pairs) * self.num_heads * 2 * (self.head_size_k + self.head_size_v)

    def qo_bytes(self) -> int:
        """Bytes of query read plus output written (fp16)."""
        return self.total_q * self.num_heads * (self.head_size_k + self.head_size_v) * 2


def _fill_normal(out: np.ndarray, seed: int, std: float, threads: int | None = None) -> None:
    """Fill a float16 array with N(0, std^2) draws, chunk-wise from child streams."""
    flat = out.reshape(-1)
    n = flat.shape[0]
    nchunks = (n + _CHUNK - 1) // _CHUNK
    kids = np.random.SeedSequence(seed).spawn(nchunks)

    def work(k: int) -> None:
        g = np.random.Generator(np.random.PCG64(kids[k]))
        lo = k * _CHUNK
        hi = min(n, lo + _CHUNK)
        v = g.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        flat[lo:hi] = v

    threads = threads or min(16, max(1, len(os.sched_getaffinity(0))))
    if nchunks == 1 or threads == 1:
        for k in range(nchunks):
            work(k)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(nchunks)))


def compress_mask(fill: float = -10000.0) -> np.ndarray:
    """The shared 2048 x 2048 fp16 causal mask of MASK_TYPE_NORM_COMPRESS.

    PagedAttentionOperation "Constraints": the strict upper triangle holds a
    large negative fill (-10000 in the op-plugin test, -60000 also allowed);
    the diagonal and the lower triangle are 0.
    """
    n = COMPRESS_MASK_SIZE
    m = np.zeros((n, n), dtype=np.float16)
    iu = np.triu_indices(n, k=1)
    m[iu] = np.float16(fill)
    return m


def alibi_slopes(num_heads: int) -> np.ndarray:
    """Per-head ALiBi slopes 2^(-8 (h+1) / H), as float32 (an input, not a rule of the kernel)."""
    h = np.arange(num_heads, dtype=np.float64)
    return np.exp2(-8.0 * (h + 1.0) / num_heads).astype(np.float32)


def norm_mask(context_lens, q_seqlens, max_kv: int, seed: int, bias_std: float = 0.5,
              fill: float = -10000.0) -> np.ndarray:
    """A MASK_TYPE_NORM tensor fp16 [B, max q, max_kv]: for query token i of
    sequence b (position p = L - q + i) and key j < L, a seeded N(0, bias_std^2)
    bias where j <= p and ``fill`` above the diagonal; entries outside the
    sequence (i >= q or j >= L) are NaN, so reading one shows up in the result."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(q_seqlens, dtype=np.int64)
    B, maxq = ctx.shape[0], int(ql.max())
    rng = np.random.default_rng(seed)
    m = np.full((B, maxq, max_kv), np.nan, dtype=np.float16)
    for b in range(B):
        L, q = int(ctx[b]), int(ql[b])
        pos = (L - q + np.arange(q))[:, None]
        j = np.arange(L)[None, :]
        bias = rng.normal(0.0, bias_std, size=(q, L))
        m[b, :q, :L] = np.where(j <= pos, bias, fill).astype(np.float16)
    return m


def make_workload(
    name: str,
    *,
    context_lens,
    q_seqlens=None,
    num_heads: int,
    kv_heads: int,
    head_size_k: int,
    head_size_v: int | None = None,
    block_size: int,
    mask_type: int = MASK_NONE,
    std: float = 1.0,
    seed: int = 0,
    spare: float = 0.10,
    num_blocks: int | None = None,
    extra_table_cols: int = 0,
    chunk_blocks: int = 0,
    mask_fill: float = -10000.0,
    poison_unused: bool = True,
    scale: float | None = None,
    shared_kv: bool = False,
) -> Workload:
    """Build one seeded workload.

    Physical blocks are a seeded random permutation of ``[0, num_blocks)``
    handed out to sequences without overlap (the GQA-decode recipe: enough
    blocks for every sequence plus ``spare`` extra). Table entries past a
    sequence's last block still hold valid random indices, as the pages require
    of every entry. Cache slots no sequence uses (the tail of each last block
    and the spare blocks) are set to NaN when ``poison_unused``, so reading one
    shows up in the result.

    ``shared_kv``: one cache holds both, V of a token being the first
    ``head_size_v`` dims of its K row (the MLA-style latent cache); the device
    run passes the K cache as the value cache, and ``value_cache`` here is the
    explicit copy of those dims that the oracle reads.
    """
    head_size_v = head_size_k if head_size_v is None else head_size_v
    assert not shared_kv or head_size_v <= head_size_k
    ctx = np.asarray(context_lens, dtype=np.int32).reshape(-1)
    B = ctx.shape[0]
    ql = (np.ones(B, dtype=np.int32) if q_seqlens is None
          else np.broadcast_to(np.asarray(q_seqlens, dtype=np.int32), (B,)).copy())
    nb_seq = (ctx.astype(np.int64) + block_size - 1) // block_size
    need = int(nb_seq.sum())
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(need * (1.0 + spare))))
    assert num_blocks >= need, "not enough physical blocks"
    maxnb = int(nb_seq.max()) + extra_table_cols
    maxnb = max(maxnb, 1)

    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = rng.integers(0, num_blocks, size=(B, maxnb), dtype=np.int32)
    off = 0
    for b in range(B):
        n = int(nb_seq[b])
        tables[b, :n] = perm[off:off + n]
        off += n

    total_q = int(ql.sum())
    query = np.empty((total_q, num_heads, head_size_k), dtype=np.float16)
    kc = np.empty((num_blocks, block_size, kv_heads, head_size_k), dtype=np.float16)
    vc = None if shared_kv else np.empty((num_blocks, block_size, kv_heads, head_size_v),
                                          dtype=np.float16)
    _fill_normal(query, seed * 7 + 1, std)
    _fill_normal(kc, seed * 7 + 2, std)
    if vc is not None:
        _fill_normal(vc, seed * 7 + 3, std)

    if poison_unused:
        used = np.zeros(num_blocks, dtype=bool)
        for b in range(B):
            n = int(nb_seq[b])
            blocks = tables[b, :n]
            used[blocks] = True
            tail = int(ctx[b]) - (n - 1) * block_size  # valid slots in the last block
            if tail < block_size:
                kc[blocks[n - 1], tail:] = np.float16(np.nan)
                if vc is not None:
                    vc[blocks[n - 1], tail:] = np.float16(np.nan)
        kc[~used] = np.float16(np.nan)
        if vc is not None:
            vc[~used] = np.float16(np.nan)
    if shared_kv:
        vc = np.ascontiguousarray(kc[..., :head_size_v])

    if mask_type == MASK_NORM_COMPRESS:
        mask = compress_mask(mask_fill)
    elif mask_type == MASK_NORM:
        mask = norm_mask(ctx, ql, maxnb * block_size, seed * 7 + 4, fill=mask_fill)
    else:
        mask = None
    slopes = alibi_slopes(num_heads) if mask_type == MASK_ALIBI else None
    if scale is None:
        scale = 1.0 / math.sqrt(head_size_k)
    return Workload(
        name=name, num_heads=num_heads, kv_heads=kv_heads, head_size_k=head_size_k,
        head_size_v=head_size_v, block_size=block_size, num_blocks=num_blocks,
        max_blocks_per_seq=maxnb, mask_type=mask_type, scale=float(scale),
        context_lens=ctx, q_seqlens=ql, block_tables=tables, query=query,
        key_cache=kc, value_cache=vc, mask=mask, alibi_slopes=slopes,
        chunk_blocks=chunk_blocks,
        meta={"seed": seed, "std": std, "shared_kv": bool(shared_kv)},
    )


# --- the five named workloads -------------------------------------------------

def tiny_decode(seed: int = 0) -> Workload:
    """Tiny decode: B=2, H=Hk=4, hk=64, bs=16, 32 blocks, L={37,100}, q=1, no mask."""
    return make_workload("tiny_decode", context_lens=[37, 100], num_heads=4, kv_heads=4,
                         head_size_k=64, block_size=16, num_blocks=32, seed=seed)


def gqa_decode(seed: int = 0, batch: int = 64, max_len: int = 4096) -> Workload:
    """GQA decode: B=64, H=32, Hk=8, hk=128, bs=128, L ~ U[1,4096], q=1, no mask."""
    rng = np.random.default_rng(seed + 1000)
    ctx = rng.integers(1, max_len + 1, size=batch, dtype=np.int32)
    return make_workload("gqa_decode", context_lens=ctx, num_heads=32, kv_heads=8,
                         head_size_k=128, block_size=128, seed=seed)


def spec_decode(seed: int = 0, batch: int = 32, max_len: int = 8192, q: int = 4) -> Workload:
    """Parallel/speculative decode: B=32, H=Hk=32, hk=128, bs=128, q=4,
    L ~ U[64,8192], compressed 2048x2048 causal mask with fill -10000."""
    rng = np.random.default_rng(seed + 2000)
    ctx = rng.integers(64, max_len + 1, size=batch, dtype=np.int32)
    return make_workload("spec_decode", context_lens=ctx, q_seqlens=q, num_heads=32,
                         kv_heads=32, head_size_k=128, block_size=128,
                         mask_type=MASK_NORM_COMPRESS, seed=seed)


def alibi_decode(seed: int = 0, batch: int = 128, max_len: int = 2048) -> Workload:
    """ALiBi decode: B=128, H=Hk=40, hk=128, bs=128, L ~ U[1,2048], q=1,
    slopes 2^(-8(h+1)/40)."""
    rng = np.random.default_rng(seed + 3000)
    ctx = rng.integers(1, max_len + 1, size=batch, dtype=np.int32)
    return make_workload("alibi_decode", context_lens=ctx, num_heads=40, kv_heads=40,
                         head_size_k=128, block_size=128, mask_type=MASK_ALIBI, seed=seed)


def mqa_split(seed: int = 0, batch: int = 8, ctx_len: int = 32768, chunk_blocks: int = 16) -> Workload:
    """Long-context MQA split-KV: B=8, H=64, Hk=1, hk=hv=512, bs=128, L=32768,
    q=1, values ~ N(0, 0.5^2), 16-block chunks."""
    return make_workload("mqa_split", context_lens=[ctx_len] * batch, num_heads=64, kv_heads=1,
                         head_size_k=512, block_size=128, std=0.5, seed=seed,
                         chunk_blocks=chunk_blocks)


def mla_decode(seed: int = 0, batch: int = 64, max_len: int = 8192) -> Workload:
    """MLA-style decode on a shared-KV latent cache: B=64, H=16, Hk=1, K rows
    of 576 dims whose first 512 are V, bs=64, L ~ U[1,8192], q=1, N(0, 0.5^2)."""
    rng = np.random.default_rng(seed + 4000)
    ctx = rng.integers(1, max_len + 1, size=batch, dtype=np.int32)
    return make_workload("mla_decode", context_lens=ctx, num_heads=16, kv_heads=1,
                         head_size_k=576, head_size_v=512, block_size=64, std=0.5, seed=seed,
                         shared_kv=True)


def prefill_causal(seed: int = 0, batch: int = 4, seq_len: int = 2048) -> Workload:
    """Prefill over the paged cache (PA_ENCODER shape, q = L): B=4, H=Hk=32,
    hk=128, bs=128, q = L = 2048, compressed causal mask with fill -10000."""
    return make_workload("prefill_causal", context_lens=[seq_len] * batch, q_seqlens=seq_len,
                         num_heads=32, kv_heads=32, head_size_k=128, block_size=128,
                         mask_type=MASK_NORM_COMPRESS, seed=seed)


NAMED = {
    "tiny_decode": tiny_decode,
    "gqa_decode": gqa_decode,
    "spec_decode": spec_decode,
    "alibi_decode": alibi_decode,
    "mqa_split": mqa_split,
    "mla_decode": mla_decode,
    "prefill_causal": prefill_causal,
}
