"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes the oracle to one of: numpy's own fp16 conversion, the numpy
brute force with the full (uncompressed) causal mask, hand-derived golden
fixtures under tests/golden/, closed forms, or exact invariants of softmax
attention. Together they fail on a dropped scale, a wrong GQA head map, a
mis-aligned mask row, a sign error in the ALiBi bias, a transposed gather or
a tail slot read past the context length.
"""
import math
import os

import numpy as np
import pytest

from paged_kv_cache_206_gb300 import workloads as W
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(name="t", seed=0, **kw):
    kw.setdefault("num_heads", 4)
    kw.setdefault("kv_heads", 2)
    kw.setdefault("head_size_k", 16)
    kw.setdefault("block_size", 16)
    return W.make_workload(name, seed=seed, **kw)


def run(oracle_mod, w, **kw):
    out, _ = oracle_mod.attention(w, **kw)
    return out


def test_half_decode_all_bit_patterns(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_double(int(b)) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))


@pytest.mark.parametrize("case", [
    dict(context_lens=[37, 100], num_heads=4, kv_heads=4, head_size_k=64),
    dict(context_lens=[1, 16, 17, 40], num_heads=8, kv_heads=2, head_size_k=32),
    dict(context_lens=[5, 33], q_seqlens=[3, 5], num_heads=4, kv_heads=4, head_size_k=16,
         mask_type=W.MASK_NORM_COMPRESS),
    dict(context_lens=[7, 29, 64], q_seqlens=[1, 4, 2], num_heads=6, kv_heads=3,
         head_size_k=16, mask_type=W.MASK_NORM_COMPRESS, block_size=32),
    dict(context_lens=[9, 50], num_heads=4, kv_heads=1, head_size_k=16,
         mask_type=W.MASK_ALIBI),
    dict(context_lens=[9, 50], q_seqlens=[2, 3], num_heads=4, kv_heads=2, head_size_k=16,
         mask_type=W.MASK_ALIBI),
    dict(context_lens=[12, 40], num_heads=4, kv_heads=2, head_size_k=32, head_size_v=16),
    dict(context_lens=[20], num_heads=2, kv_heads=2, head_size_k=16, scale=0.37),
    dict(context_lens=[9, 50], num_heads=4, kv_heads=2, head_size_k=16,
         mask_type=W.MASK_NORM),
    dict(context_lens=[6, 33, 70], q_seqlens=[3, 1, 4], num_heads=6, kv_heads=3,
         head_size_k=16, mask_type=W.MASK_NORM, block_size=32),
    # the MLA shape: 576-dim K rows whose first 512 dims are V (shared cache)
    dict(context_lens=[5, 70], num_heads=4, kv_heads=1, head_size_k=576, head_size_v=512,
         shared_kv=True, std=0.5),
    # prefill-shaped rows (q = L) with the compressed mask, 64-dim heads
    dict(context_lens=[40, 17], q_seqlens=[40, 17], num_heads=2, kv_heads=2, head_size_k=64,
         mask_type=W.MASK_NORM_COMPRESS),
])
def test_oracle_matches_brute_force(oracle_mod, case):
    w = small(**case)
    got = run(oracle_mod, w)
    ref = brute.attention(w)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_compressed_mask_equals_full_causal_mask(oracle_mod):
    """Compressed 2048x2048 mask with the shift == full causal mask of any length."""
    for L in (1, 2047, 2048, 2049, 8192):
        for q in (1, 4, 16):
            if q > L:
                continue
            w = small(context_lens=[L], q_seqlens=[q], num_heads=2, kv_heads=1,
                      mask_type=W.MASK_NORM_COMPRESS, block_size=128, seed=L + q)
            np.testing.assert_allclose(run(oracle_mod, w), brute.attention(w), rtol=0,
                                       atol=1e-12, err_msg=f"L={L} q={q}")


def test_mask_alignment_golden(oracle_mod):
    """Zero queries make every visible score equal; V encodes the key index, so
    the output reveals the set 0..p each query row sees."""
    rows = [tuple(map(int, ln.split())) for ln in open(os.path.join(GOLDEN, "mask_alignment.txt"))
            if ln.strip() and not ln.startswith("#")]
    for L, q, i, p in rows:
        w = small(context_lens=[L], q_seqlens=[q], num_heads=1, kv_heads=1,
                  mask_type=W.MASK_NORM_COMPRESS, block_size=64, poison_unused=False)
        w.query[:] = 0
        w.value_cache[:] = 0
        j = np.arange(L)
        phys = w.block_tables[0][j // w.block_size]
        slot = j % w.block_size
        w.value_cache[phys, slot, 0, 0] = (j & 63).astype(np.float16)
        w.value_cache[phys, slot, 0, 1] = ((j >> 6) & 63).astype(np.float16)
        w.value_cache[phys, slot, 0, 2] = (j >> 12).astype(np.float16)
        out = run(oracle_mod, w)[i, 0, :3]
        vis = np.arange(p + 1)
        exp = [np.mean(vis & 63), np.mean((vis >> 6) & 63), np.mean(vis >> 12)]
        np.testing.assert_allclose(out, exp, rtol=0, atol=1e-9, err_msg=f"L={L} q={q} i={i}")


def test_uniform_golden(oracle_mod):
    text = [ln.split() for ln in open(os.path.join(GOLDEN, "tiny_uniform.txt"))
            if ln.strip() and not ln.startswith("#")]
    k = 0
    n = 0
    while k < len(text):
        assert text[k][0] == "case"
        L = int(text[k][1])
        vals = np.array([[float(x) for x in r] for r in text[k + 1:k + 1 + L]])
        expect = np.array([float(x) for x in text[k + 1 + L][1:]])
        k += L + 2
        w = small(context_lens=[L], num_heads=1, kv_heads=1, seed=L)
        w.query[:] = 0
        j = np.arange(L)
        phys = w.block_tables[0][j // w.block_size]
        w.value_cache[phys, j % w.block_size, 0, :] = 0
        w.value_cache[phys, j % w.block_size, 0, :4] = vals.astype(np.float16)
        out = run(oracle_mod, w)[0, 0]
        np.testing.assert_allclose(out[:4], expect, rtol=0, atol=1e-12)
        assert np.all(out[4:] == 0)
        n += 1
    assert n == 3


def test_block_permutation_invariance(oracle_mod):
    """Moving physical blocks and rewriting the table changes nothing, bit for bit."""
    w = small(context_lens=[30, 77, 3], q_seqlens=[2, 1, 3], mask_type=W.MASK_NORM_COMPRESS,
              seed=3)
    ref = run(oracle_mod, w)
    rng = np.random.default_rng(11)
    perm = rng.permutation(w.num_blocks)  # new home of each old block
    kc = np.empty_like(w.key_cache)
    vc = np.empty_like(w.value_cache)
    kc[perm] = w.key_cache
    vc[perm] = w.value_cache
    w.key_cache, w.value_cache = kc, vc
    w.block_tables = perm[w.block_tables].astype(np.int32)
    assert np.array_equal(run(oracle_mod, w), ref)


def test_identical_keys_give_mean_of_visible_values(oracle_mod):
    w = small(context_lens=[11, 40], q_seqlens=[3, 4], num_heads=2, kv_heads=1,
              mask_type=W.MASK_NORM_COMPRESS, seed=5)
    w.key_cache[:] = w.key_cache[w.block_tables[0][0], 0, 0]
    out = run(oracle_mod, w)
    qs = 0
    for b in range(w.batch):
        L, q = int(w.context_lens[b]), int(w.q_seqlens[b])
        j = np.arange(L)
        V = w.value_cache[w.block_tables[b][j // w.block_size], j % w.block_size, 0].astype(np.float64)
        for i in range(q):
            p = L - q + i
            for h in range(2):
                np.testing.assert_allclose(out[qs + i, h], V[:p + 1].mean(0), rtol=0, atol=1e-12)
        qs += q


def test_single_token_context_returns_v0(oracle_mod):
    w = small(context_lens=[1, 1], num_heads=4, kv_heads=2, seed=8)
    out = run(oracle_mod, w)
    for b in range(2):
        for h in range(4):
            v0 = w.value_cache[w.block_tables[b][0], 0, h // 2].astype(np.float64)
            assert np.array_equal(out[b, h], v0)


def test_q1_causal_mask_equals_no_mask(oracle_mod):
    w = small(context_lens=[1, 19, 2049], num_heads=2, kv_heads=2, block_size=64,
              mask_type=W.MASK_NORM_COMPRESS, seed=9)
    a = run(oracle_mod, w)
    w.mask_type, w.mask = W.MASK_NONE, None
    assert np.array_equal(a, run(oracle_mod, w))


def test_gqa_equals_mha_with_repeated_kv(oracle_mod):
    """kvh = h / G: GQA equals MHA whose kv head h holds the GQA kv head h // G."""
    w = small(context_lens=[13, 50], q_seqlens=[2, 1], num_heads=6, kv_heads=2, seed=12,
              mask_type=W.MASK_NORM_COMPRESS)
    gqa = run(oracle_mod, w)
    G = 3
    w.key_cache = np.repeat(w.key_cache, G, axis=2)
    w.value_cache = np.repeat(w.value_cache, G, axis=2)
    w.kv_heads = 6
    assert np.array_equal(run(oracle_mod, w), gqa)


def test_alibi_zero_slope_equals_no_mask(oracle_mod):
    w = small(context_lens=[17, 40], q_seqlens=[1, 3], mask_type=W.MASK_ALIBI, seed=13)
    w.alibi_slopes[:] = 0
    a = run(oracle_mod, w)
    w.mask_type, w.alibi_slopes = W.MASK_NONE, None
    assert np.array_equal(a, run(oracle_mod, w))


def test_alibi_identical_keys_closed_form(oracle_mod):
    """Identical keys, q = 1: weights w_j ~ r^(L-1-j), r = exp(-slope) (a geometric series)."""
    L = 45
    w = small(context_lens=[L], num_heads=4, kv_heads=4, mask_type=W.MASK_ALIBI, seed=14)
    w.key_cache[:] = w.key_cache[w.block_tables[0][0], 0]
    out = run(oracle_mod, w)
    j = np.arange(L)
    for h in range(4):
        V = w.value_cache[w.block_tables[0][j // w.block_size], j % w.block_size, h].astype(np.float64)
        r = math.exp(-float(w.alibi_slopes[h]))
        wts = r ** (L - 1 - j)
        denom = (1 - r ** L) / (1 - r)
        np.testing.assert_allclose(wts.sum(), denom, rtol=1e-13)
        np.testing.assert_allclose(out[0, h], (wts[:, None] * V).sum(0) / denom, rtol=0, atol=1e-12)


def test_tail_slots_and_spare_blocks_never_read(oracle_mod):
    """The generator fills unused slots with NaN; any read would poison the output."""
    w = small(context_lens=[3, 17, 31], q_seqlens=[1, 2, 3], mask_type=W.MASK_NORM_COMPRESS,
              seed=15)
    assert np.isnan(w.key_cache.astype(np.float32)).any()
    assert np.isfinite(run(oracle_mod, w)).all()


def test_subset_computes_only_listed_sequences(oracle_mod):
    w = small(context_lens=[10, 20, 30], q_seqlens=[1, 2, 1], seed=16)
    full = run(oracle_mod, w)
    sub, used = oracle_mod.attention(w, subset=[2, 0], threads=2)
    assert np.array_equal(sub[[0, 3]], full[[0, 3]])
    assert np.all(sub[1:3] == 0)
    assert 1 <= used <= 2


def _causal_norm(w, bias_std):
    """Replace w's NORM mask by one with the given bias spread (0: a plain causal mask)."""
    w.mask = W.norm_mask(w.context_lens, w.q_seqlens, w.max_blocks_per_seq * w.block_size,
                         seed=99, bias_std=bias_std)
    return w


def test_norm_causal_mask_equals_compressed_mask(oracle_mod):
    """A per-sequence NORM mask holding the plain causal mask gives what the
    compressed 2048 x 2048 mask gives, below and past 2048 keys."""
    for L, q in ((1, 1), (40, 4), (2048, 3), (2049, 2), (3000, 5)):
        w = small(context_lens=[L, 17], q_seqlens=[q, 1], num_heads=2, kv_heads=1,
                  block_size=64, mask_type=W.MASK_NORM, seed=L)
        norm = run(oracle_mod, _causal_norm(w, 0.0))
        w.mask_type, w.mask = W.MASK_NORM_COMPRESS, W.compress_mask()
        np.testing.assert_array_equal(norm, run(oracle_mod, w), err_msg=f"L={L} q={q}")


def test_norm_bias_is_read_per_sequence_and_token(oracle_mod):
    """A bias on one (sequence, query token, key) entry changes exactly that
    output row: a transposed or mis-strided read would move it."""
    w = small(context_lens=[30, 45], q_seqlens=[2, 3], num_heads=2, kv_heads=2,
              mask_type=W.MASK_NORM, seed=21)
    w = _causal_norm(w, 0.0)
    base = run(oracle_mod, w)
    w.mask[1, 2, 7] = np.float16(3.0)  # sequence 1, query token 2 (global row 4), key 7
    got = run(oracle_mod, w)
    changed = np.abs(got - base).max(axis=(1, 2)) > 0
    assert changed.tolist() == [False, False, False, False, True]
