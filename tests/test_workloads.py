"""The seeded input generator: the layout facts the GPU runs rely on."""
import numpy as np

from paged_kv_cache_206_gb300 import workloads as W


def test_shared_kv_value_is_the_leading_dims_of_each_key_row():
    w = W.make_workload("s", context_lens=[70, 5], num_heads=4, kv_heads=2, head_size_k=96,
                        head_size_v=64, block_size=16, seed=3, shared_kv=True)
    assert w.shared_kv
    np.testing.assert_array_equal(w.value_cache.view(np.uint16),
                                  w.key_cache[..., :64].view(np.uint16))  # NaN-safe compare
    # unique bytes: the K rows only
    assert w.kv_bytes() == 75 * 2 * 96 * 2


def test_separate_caches_count_both():
    w = W.make_workload("d", context_lens=[70, 5], num_heads=4, kv_heads=2, head_size_k=96,
                        head_size_v=64, block_size=16, seed=3)
    assert not w.shared_kv
    assert w.kv_bytes() == 75 * 2 * (96 + 64) * 2


def test_unused_slots_are_poisoned_and_tables_do_not_overlap():
    w = W.make_workload("p", context_lens=[37, 100], num_heads=2, kv_heads=2, head_size_k=64,
                        block_size=16, seed=4)
    nb = [3, 7]
    used = np.concatenate([w.block_tables[b, :nb[b]] for b in range(2)])
    assert len(set(used.tolist())) == len(used)
    assert np.isnan(w.key_cache[w.block_tables[0, 2], 37 - 32:].astype(np.float32)).all()
    assert np.isfinite(w.key_cache[w.block_tables[0, 2], :37 - 32].astype(np.float32)).all()
    spare = np.setdiff1d(np.arange(w.num_blocks), used)
    assert np.isnan(w.value_cache[spare].astype(np.float32)).all()


def test_norm_mask_layout_and_poison():
    m = W.norm_mask([5, 3], [2, 1], max_kv=8, seed=1)
    assert m.shape == (2, 2, 8) and m.dtype == np.float16
    # sequence 0: L=5, q=2 -> positions 3, 4; key 4 is masked for token 0 only
    assert m[0, 0, 4] == np.float16(-10000.0) and np.isfinite(m[0, 1, 4])
    assert np.isnan(m[0, :, 5:].astype(np.float32)).all()
    assert np.isnan(m[1, 1].astype(np.float32)).all()  # sequence 1 has one query token


def test_attention_flops_count_the_visible_keys():
    # causal: L=5, q=3 -> rows see 3, 4, 5 keys = 12 pairs; L=4, q=1 -> 4
    w = W.make_workload("f", context_lens=[5, 4], q_seqlens=[3, 1], num_heads=2, kv_heads=1,
                        head_size_k=16, block_size=16, mask_type=W.MASK_NORM_COMPRESS, seed=5)
    assert w.attn_flops() == 16 * 2 * 2 * 32
    w.mask_type = W.MASK_NONE  # every row sees all L keys: 3*5 + 4 = 19
    assert w.attn_flops() == 19 * 2 * 2 * 32
