"""Brute-force paged attention in numpy float64, for tiny inputs.

A second, independent statement of the operation that pins the oracle: it
resolves the block table with numpy fancy indexing, widens fp16 with numpy's
own conversion, and applies the causal mask in its FULL form (a [q, L] slice of
the L x L causal mask: 0 on and below the diagonal, the fill above it) rather
than through the compressed 2048 x 2048 tensor and its shift. Source of the
definitions: PagedAttentionOperation, "Constraints" (block tables, context
lengths that include the query tokens, prefix = max(0, kvSeqLen - qSeqLen),
the causal mask and its fill value, GQA).
"""
import numpy as np

MASK_NONE, MASK_NORM, MASK_ALIBI, MASK_NORM_COMPRESS = 0, 1, 2, 5


def full_causal_rows(L, q, fill):
    """Rows L-q .. L-1 of the L x L causal mask (0 where key <= row, else fill)."""
    rows = np.arange(L - q, L)[:, None]
    cols = np.arange(L)[None, :]
    return np.where(cols <= rows, 0.0, float(np.float16(fill)))


def attention(w, mask_fill=-10000.0):
    """float64 [sum q, H, hv]; the compressed mask is replaced by the full causal mask."""
    H, Hk = w.num_heads, w.kv_heads
    G = H // Hk
    out = np.zeros((w.total_q, H, w.head_size_v))
    qs = 0
    for b in range(w.batch):
        L, q = int(w.context_lens[b]), int(w.q_seqlens[b])
        j = np.arange(L)
        phys = w.block_tables[b][j // w.block_size]
        K = w.key_cache[phys, j % w.block_size].astype(np.float64)    # [L, Hk, hk]
        V = w.value_cache[phys, j % w.block_size].astype(np.float64)  # [L, Hk, hv]
        Q = w.query[qs:qs + q].astype(np.float64)                     # [q, H, hk]
        for h in range(H):
            kv = h // G
            S = w.scale * (Q[:, h, :] @ K[:, kv, :].T)                 # [q, L]
            if w.mask_type == MASK_NORM_COMPRESS:
                S = S + full_causal_rows(L, q, mask_fill)
            elif w.mask_type == MASK_NORM:
                S = S + w.mask[b, :q, :L].astype(np.float64)
            elif w.mask_type == MASK_ALIBI:
                pos = (L - q + np.arange(q))[:, None]
                S = S + float(w.alibi_slopes[h]) * (j[None, :] - pos)
            S = S - S.max(axis=1, keepdims=True)
            P = np.exp(S)
            P /= P.sum(axis=1, keepdims=True)
            out[qs:qs + q, h, :] = P @ V[:, kv, :]
        qs += q
    return out
