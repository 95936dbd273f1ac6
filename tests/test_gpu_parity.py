"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Tolerance (fp16 outputs of O(1) magnitude, fp32 accumulation on the GPU,
float64 in the oracle): max |gpu - oracle| <= 1e-2 and mean |gpu - oracle| <=
1e-3 over every compared element. The work list is compared bit for bit with
the oracle's planner in tests/test_plan.py; here the kernels run the list that
pa_plan builds.

Small cases run the oracle on every output element; they still span several
16-token sub-tiles, several KV blocks per split, ragged last blocks and both
split and unsplit items. The full-size workloads run on the GPU exactly as the
benchmark launches them (automatic chunking for the device's SM count, 16-block
chunks for the long-context MQA case) and compare sampled sequences.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import paged_kv_cache_206_gb300 as pa
from paged_kv_cache_206_gb300 import build_lib
from paged_kv_cache_206_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3
CORES = max(1, len(os.sched_getaffinity(0)))


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.build()
    pa.load_library()


def run_gpu(w, chunk_blocks=None):
    db = pa.DeviceBatch(w, chunk_blocks=chunk_blocks)
    out = db.forward()
    st, bits = db.status()
    assert st == pa.PA_OK, (pa.status_string(st), bits)
    return out.float().cpu().numpy().astype(np.float64), db


def compare(got, ref, rows=None):
    if rows is not None:
        got, ref = got[rows], ref[rows]
    assert np.isfinite(got).all(), "non-finite GPU output"
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS, f"max abs err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"mean abs err {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def full_parity(oracle_mod, w, chunk_blocks=None):
    got, db = run_gpu(w, chunk_blocks)
    ref, _ = oracle_mod.attention(w, threads=CORES)
    return compare(got, ref), db


# ---- small cases: every element against the oracle -------------------------

CASES = {
    "tiny_decode": lambda: W.tiny_decode(),
    "gqa_small": lambda: W.gqa_decode(batch=8, max_len=1000, seed=1),
    "spec_small": lambda: W.spec_decode(batch=4, max_len=2600, seed=2),
    "alibi_small": lambda: W.alibi_decode(batch=6, max_len=700, seed=3),
    "mqa8_hd512": lambda: W.make_workload("mqa8", context_lens=[700, 1500, 33], num_heads=8,
                                          kv_heads=1, head_size_k=512, block_size=64, std=0.5,
                                          seed=4),
    "hk576_hv512": lambda: W.make_workload("mla", context_lens=[300, 77], num_heads=4,
                                           kv_heads=1, head_size_k=576, head_size_v=512,
                                           block_size=64, seed=5),
    "hk96": lambda: W.make_workload("hk96", context_lens=[129, 40, 300], num_heads=6,
                                    kv_heads=2, head_size_k=96, block_size=32, seed=6),
    "hk80_hv48": lambda: W.make_workload("hk80", context_lens=[50, 211], num_heads=2,
                                         kv_heads=2, head_size_k=80, head_size_v=48,
                                         block_size=16, seed=7),
    # value heads of 17-31 eight-dim chunks (144-240 dims) on the CUDA-core
    # kernel: one lane per chunk (found by the random shapes, where 16 lanes
    # left dims 128 and up unaccumulated)
    "hk192_shared_alibi": lambda: W.make_workload("hk192", context_lens=[418, 99], num_heads=2,
                                                  kv_heads=2, head_size_k=192, block_size=48,
                                                  mask_type=W.MASK_ALIBI, shared_kv=True,
                                                  seed=8, chunk_blocks=2),
    "hk160_hv224": lambda: W.make_workload("hk160", context_lens=[300, 77, 129], num_heads=6,
                                           kv_heads=3, head_size_k=160, head_size_v=224,
                                           block_size=32, seed=9),
    "hk256_g8": lambda: W.make_workload("g8", context_lens=[1, 2, 15, 16, 17, 255, 256, 257],
                                        num_heads=16, kv_heads=2, head_size_k=256,
                                        block_size=128, seed=8),
    "g2_q3_mask": lambda: W.make_workload("g2q3", context_lens=[3, 4, 20, 129, 2047, 2048, 2049,
                                                               3000],
                                          q_seqlens=3, num_heads=4, kv_heads=2,
                                          head_size_k=64, block_size=32,
                                          mask_type=W.MASK_NORM_COMPRESS, seed=9),
    "q_ragged_mask": lambda: W.make_workload("qr", context_lens=[5, 64, 300, 2100, 9],
                                             q_seqlens=[1, 8, 3, 5, 8], num_heads=1,
                                             kv_heads=1, head_size_k=128, block_size=64,
                                             mask_type=W.MASK_NORM_COMPRESS, seed=10),
    "mask_60000": lambda: W.make_workload("m6", context_lens=[40, 2200], q_seqlens=4,
                                          num_heads=2, kv_heads=2, head_size_k=128,
                                          block_size=128, mask_type=W.MASK_NORM_COMPRESS,
                                          mask_fill=-60000.0, seed=11),
    "alibi_q2_gqa": lambda: W.make_workload("aq", context_lens=[9, 300, 1000], q_seqlens=2,
                                            num_heads=8, kv_heads=2, head_size_k=128,
                                            block_size=16, mask_type=W.MASK_ALIBI, seed=12),
    "bs16_long": lambda: W.make_workload("bs16", context_lens=[4000, 1, 17], num_heads=4,
                                         kv_heads=4, head_size_k=128, block_size=16, seed=13),
    # MASK_TYPE_NORM: a per-sequence [q, L] additive mask (NaN outside the
    # sequence, so a read past q or L shows): CUDA-core, mma.sync paths
    "norm_q1": lambda: W.make_workload("n1", context_lens=[70, 513, 1], num_heads=3, kv_heads=3,
                                       head_size_k=128, block_size=32, mask_type=W.MASK_NORM,
                                       seed=17),
    "norm_spec_gqa": lambda: W.make_workload("n2", context_lens=[40, 900, 3], q_seqlens=[3, 2, 3],
                                             num_heads=4, kv_heads=2, head_size_k=128,
                                             block_size=64, mask_type=W.MASK_NORM, seed=18),
    # shared-KV caches on the warp-pipelined kernels (V read from the K boxes):
    # mma.sync with 576/512 and 4 rows, CUDA-core with 64-wide and 16-wide boxes
    "mma_mla_shared": lambda: W.make_workload("mmas", context_lens=[900, 77, 16], num_heads=4,
                                              kv_heads=1, head_size_k=576, head_size_v=512,
                                              block_size=64, std=0.5, seed=14, shared_kv=True),
    "fma_shared_hd128": lambda: W.make_workload("fs", context_lens=[333, 40], num_heads=2,
                                                kv_heads=2, head_size_k=128, head_size_v=64,
                                                block_size=32, seed=15, shared_kv=True),
    "fma_shared_hk96": lambda: W.make_workload("fs96", context_lens=[129, 500], num_heads=3,
                                               kv_heads=3, head_size_k=96, head_size_v=48,
                                               block_size=16, seed=16, shared_kv=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_small_parity(oracle_mod, name):
    full_parity(oracle_mod, CASES[name]())


@pytest.mark.parametrize("chunk", [1, 2, 5, 1000])
def test_chunking_does_not_change_the_result(oracle_mod, chunk):
    w = W.gqa_decode(batch=6, max_len=1500, seed=20)
    (mx, mean), db = full_parity(oracle_mod, w, chunk_blocks=chunk)
    if chunk == 1:
        assert db.plan.combine.shape[0] > 0
    if chunk == 1000:
        assert db.plan.combine.shape[0] == 0


def test_split_and_unsplit_agree(oracle_mod):
    w = W.spec_decode(batch=3, max_len=3000, seed=21)
    a, _ = run_gpu(w, chunk_blocks=1)
    b, _ = run_gpu(w, chunk_blocks=100)
    compare(a, b)


def test_repeat_runs_are_identical():
    w = W.gqa_decode(batch=8, max_len=2000, seed=22)
    db = pa.DeviceBatch(w)
    a = db.forward().clone()
    b = db.forward().clone()
    assert torch.equal(a, b)


def test_block_index_out_of_range_is_reported():
    """A table entry outside [0, num_blocks) is flagged by the kernel's own bounds
    check and never dereferenced; the other sequences are unaffected."""
    w = W.gqa_decode(batch=4, max_len=600, seed=23)
    good = pa.DeviceBatch(w, chunk_blocks=1000)
    ref = good.forward().clone()
    w.block_tables[2, 0] = w.num_blocks + 5
    bad = pa.DeviceBatch(w, chunk_blocks=1000)
    out = bad.forward()
    st, bits = bad.status()
    assert st == pa.PA_ERR_BLOCK_INDEX and bits & 1
    keep = np.ones(w.total_q, bool)
    keep[2] = False
    assert torch.equal(out[torch.from_numpy(keep).cuda()], ref[torch.from_numpy(keep).cuda()])
    pa.pa_status_clear(bad.workspace)
    assert bad.status()[0] == pa.PA_OK


# ---- 64-row tiles (tcgen05 kernel) -------------------------------------------

TC_CASES = {
    # 16 rows, bs=16: a 128-token tile gathers 8 blocks; ragged last tile
    "tc_r16_bs16": lambda: W.make_workload("r16", context_lens=[100, 300, 17, 129], num_heads=16,
                                           kv_heads=1, head_size_k=128, block_size=16, seed=30),
    # the long-context MQA shape, shortened: 64 heads on one kv head of 512 dims
    "tc_mqa_hd512": lambda: W.make_workload("mqa", context_lens=[2085, 700, 128, 1], num_heads=64,
                                            kv_heads=1, head_size_k=512, block_size=128,
                                            std=0.5, seed=31, chunk_blocks=4),
    # 64 rows = GQA 16 x 4 speculative tokens, compressed causal mask past 2048
    "tc_spec_mask": lambda: W.make_workload("tcm", context_lens=[2200, 64, 700], q_seqlens=4,
                                            num_heads=32, kv_heads=2, head_size_k=128,
                                            block_size=64, mask_type=W.MASK_NORM_COMPRESS, seed=32),
    # ALiBi with 24 rows on hk=256
    "tc_alibi_hd256": lambda: W.make_workload("tca", context_lens=[300, 1000], num_heads=24,
                                              kv_heads=1, head_size_k=256, block_size=32,
                                              mask_type=W.MASK_ALIBI, seed=33),
    # 128 rows per (b, kv head): two row tiles, ragged q
    "tc_two_tiles": lambda: W.make_workload("tc2", context_lens=[500, 130], q_seqlens=[4, 3],
                                            num_heads=32, kv_heads=1, head_size_k=128,
                                            block_size=128, mask_type=W.MASK_NORM_COMPRESS, seed=34),
    # block_size 256: a tile is half a block
    "tc_bs256": lambda: W.make_workload("tc256", context_lens=[600, 256, 257], num_heads=16,
                                        kv_heads=1, head_size_k=128, block_size=256, seed=35),
    # prefill (q = L) with the causal mask: row tiles skip the keys past their
    # last token; 1-block chunks make splits that lie wholly past it (empty,
    # weight zero in the combine)
    "tc_prefill_split": lambda: W.make_workload("pf", context_lens=[300, 129], q_seqlens=[300, 129],
                                                num_heads=2, kv_heads=2, head_size_k=128,
                                                block_size=64, mask_type=W.MASK_NORM_COMPRESS,
                                                seed=40, chunk_blocks=1),
    "tc_prefill_gqa": lambda: W.make_workload("pfg", context_lens=[200, 77], q_seqlens=[200, 70],
                                              num_heads=8, kv_heads=2, head_size_k=128,
                                              block_size=32, mask_type=W.MASK_NORM_COMPRESS,
                                              seed=41),
    # 128-row tiles (65-128 rows per kv head): causal prefill of up to 128
    # tokens, and 64-dim heads with ALiBi; every other prefill case here has
    # more than 128 rows and runs as 256-row tiles (two query tiles per CTA)
    "pf128_prefill": lambda: W.make_workload("pf128", context_lens=[100, 300, 128],
                                             q_seqlens=[100, 128, 128], num_heads=3, kv_heads=3,
                                             head_size_k=128, block_size=64,
                                             mask_type=W.MASK_NORM_COMPRESS, seed=45),
    "pf128_hd64_alibi": lambda: W.make_workload("pf128a", context_lens=[77, 400], q_seqlens=[50, 64],
                                                num_heads=4, kv_heads=2, head_size_k=64,
                                                block_size=16, mask_type=W.MASK_ALIBI, seed=46),
    # a 256-row tile whose second query tile holds only part of the rows, with
    # the causal mask past 2048 (L = 2300, q = 200)
    "pf256_ragged_long": lambda: W.make_workload("pf256", context_lens=[2300, 60], q_seqlens=[200, 60],
                                                 num_heads=2, kv_heads=2, head_size_k=128,
                                                 block_size=128, mask_type=W.MASK_NORM_COMPRESS,
                                                 seed=47),
    # many-row tiles (prefill kernel): head size 64, ALiBi, 16-token blocks
    "pf_hd64_alibi_bs16": lambda: W.make_workload("pf64", context_lens=[333, 90], q_seqlens=[40, 90],
                                                  num_heads=8, kv_heads=4, head_size_k=64,
                                                  block_size=16, mask_type=W.MASK_ALIBI, seed=42),
    # MASK_TYPE_NORM on the prefill kernel (q = 100 of L = 260, 2 heads per kv head)
    "pf_norm": lambda: W.make_workload("pfn", context_lens=[260, 100], q_seqlens=[100, 60],
                                       num_heads=4, kv_heads=2, head_size_k=128, block_size=32,
                                       mask_type=W.MASK_NORM, seed=43),
    # no mask, splits across 128-token tiles, shared-KV cache (V = K)
    "pf_shared_split": lambda: W.make_workload("pfs", context_lens=[700, 1300], q_seqlens=[70, 33],
                                               num_heads=4, kv_heads=2, head_size_k=128,
                                               block_size=64, seed=44, shared_kv=True,
                                               chunk_blocks=4),
    # MASK_TYPE_NORM on the tensor-core path: 16 heads x 2 tokens per kv head
    "tc_norm": lambda: W.make_workload("tcn", context_lens=[300, 1200], q_seqlens=[2, 1],
                                       num_heads=16, kv_heads=1, head_size_k=128, block_size=64,
                                       mask_type=W.MASK_NORM, seed=39, chunk_blocks=6),
    # 16-row tcgen05 tiles of 256/512-dim heads with separate caches:
    # 12 rows, 256-dim heads, ALiBi, 32-token blocks
    "tc_r12_hd256_alibi": lambda: W.make_workload("w256", context_lens=[333, 1000, 17], num_heads=24,
                                                kv_heads=2, head_size_k=256, block_size=32,
                                                mask_type=W.MASK_ALIBI, seed=49, chunk_blocks=3),
    # 8 heads x 2 tokens, 512-dim heads, MASK_TYPE_NORM, 16-token blocks
    "tc_r16_hd512_norm_q2": lambda: W.make_workload("w512", context_lens=[300, 90], q_seqlens=[2, 1],
                                                  num_heads=8, kv_heads=1, head_size_k=512,
                                                  block_size=16, std=0.5, mask_type=W.MASK_NORM,
                                                  seed=50, chunk_blocks=7),
    # 9-16 rows over a shared-KV cache run on the 16-row warp-level MMA kernel:
    # hk = hv = 512 shared, 16 rows, 32-token blocks (two pieces a tile)
    "wide_hd512_shared": lambda: W.make_workload("ws512", context_lens=[777, 64, 1], num_heads=16,
                                                 kv_heads=1, head_size_k=512, block_size=32,
                                                 std=0.5, seed=53, shared_kv=True, chunk_blocks=5),
    # hk = hv = 256 shared, 12 rows of two kv heads, ALiBi, 128-token blocks
    "wide_hd256_shared_alibi": lambda: W.make_workload("ws256", context_lens=[1000, 200], num_heads=24,
                                                       kv_heads=2, head_size_k=256, block_size=128,
                                                       mask_type=W.MASK_ALIBI, seed=54,
                                                       shared_kv=True, chunk_blocks=3),
    # 4 heads x 4 tokens of the shared latent cache, compressed causal mask past
    # 2048 keys (sigma > 0), 48-token blocks
    "wide_mla_causal_bs48": lambda: W.make_workload("wmc", context_lens=[2500, 70], q_seqlens=4,
                                                    num_heads=4, kv_heads=1, head_size_k=576,
                                                    head_size_v=512, block_size=48, std=0.5,
                                                    mask_type=W.MASK_NORM_COMPRESS, seed=51,
                                                    shared_kv=True, chunk_blocks=9),
    # 16 rows, shared latent cache, 96-token blocks (32-token boxes), one short sequence
    "wide_mla_bs96": lambda: W.make_workload("wm96", context_lens=[1000, 5], num_heads=16,
                                             kv_heads=1, head_size_k=576, head_size_v=512,
                                             block_size=96, std=0.5, seed=52, shared_kv=True),
    # MLA-style shared-KV cache: K rows of 576 dims, V = their first 512
    "tc_mla_shared": lambda: W.make_workload("mla", context_lens=[700, 1500, 65], num_heads=16,
                                             kv_heads=1, head_size_k=576, head_size_v=512,
                                             block_size=64, std=0.5, seed=36, shared_kv=True,
                                             chunk_blocks=8),
    # 576/512 with separate caches and two kv heads: the half-slot of kv head
    # 0 reads kv head 1's first dims, that of kv head 1 reads past the tensor
    "tc_hk576_two_heads": lambda: W.make_workload("tc576", context_lens=[300, 129], num_heads=32,
                                                  kv_heads=2, head_size_k=576, head_size_v=512,
                                                  block_size=128, std=0.5, seed=37),
    # block sizes that neither divide nor are a multiple of the key tile: the
    # boxes are the largest power of two dividing the block, so none crosses
    # into the next physical block (64-token tiles: 48 -> 16, 96 -> 32;
    # 128-token tiles: 80 -> 16, 48 -> 16)
    "tc_bs48": lambda: W.make_workload("tc48", context_lens=[300, 1000, 47], num_heads=16,
                                       kv_heads=1, head_size_k=128, block_size=48, seed=45,
                                       chunk_blocks=5),
    "tc_bs96_g64": lambda: W.make_workload("tc96", context_lens=[500, 97], num_heads=64,
                                           kv_heads=1, head_size_k=128, block_size=96, seed=46),
    "pf_bs80": lambda: W.make_workload("pf80", context_lens=[400, 250], q_seqlens=[16, 12],
                                       num_heads=8, kv_heads=1, head_size_k=128, block_size=80,
                                       mask_type=W.MASK_NORM_COMPRESS, seed=47),
    "pf_pair_bs48": lambda: W.make_workload("pp48", context_lens=[700, 330], q_seqlens=[300, 330],
                                            num_heads=4, kv_heads=2, head_size_k=128,
                                            block_size=48, mask_type=W.MASK_NORM_COMPRESS,
                                            seed=48),
    # 576/512 shared with 16-token blocks: the half slot moves as one box per block
    "tc_mla_bs16": lambda: W.make_workload("mla16", context_lens=[200, 33], num_heads=64,
                                           kv_heads=1, head_size_k=576, head_size_v=512,
                                           block_size=16, std=0.5, seed=38, shared_kv=True),
}


@pytest.mark.parametrize("name", sorted(TC_CASES))
def test_tensor_core_parity(oracle_mod, name):
    full_parity(oracle_mod, TC_CASES[name]())


# More than 32 splits of one tile (1-block chunks over long sequences): the
# combine's second round of partial-row loads and its weights past the 32 that
# a warp's lanes hold, in its 4-dims-a-lane form (value heads of 128) and its
# 8-dims-a-lane form (256 and 512), after each kernel family's fp16 partials.
SPLIT_CASES = {
    "fma_hd128_bs16": lambda: W.make_workload("s1", context_lens=[700, 20], num_heads=2,
                                              kv_heads=2, head_size_k=128, block_size=16,
                                              seed=60, chunk_blocks=1),
    "mma_hd128_gqa": lambda: W.make_workload("s2", context_lens=[5000, 130], num_heads=8,
                                             kv_heads=2, head_size_k=128, block_size=128,
                                             seed=61, chunk_blocks=1),
    "tc_mqa_hd512": lambda: W.make_workload("s3", context_lens=[4300, 300], num_heads=64,
                                            kv_heads=1, head_size_k=512, block_size=128,
                                            std=0.5, seed=62, chunk_blocks=1),
    "wide_hd256_shared": lambda: W.make_workload("s4", context_lens=[2500, 70], num_heads=16,
                                                 kv_heads=1, head_size_k=256, block_size=64,
                                                 seed=63, chunk_blocks=1, shared_kv=True),
    "wide_mla_shared": lambda: W.make_workload("s5", context_lens=[2200, 33], num_heads=16,
                                               kv_heads=1, head_size_k=576, head_size_v=512,
                                               block_size=64, seed=64, chunk_blocks=1,
                                               shared_kv=True),
}


@pytest.mark.parametrize("name", sorted(SPLIT_CASES))
def test_many_splits_parity(oracle_mod, name):
    _, db = full_parity(oracle_mod, SPLIT_CASES[name]())
    assert int(np.asarray(db.plan.combine)[:, 3].max()) > 32


def test_tensor_core_split_and_unsplit_agree(oracle_mod):
    w = TC_CASES["tc_mqa_hd512"]()
    a, _ = run_gpu(w, chunk_blocks=1)
    b, _ = run_gpu(w, chunk_blocks=100)
    compare(a, b)


def test_tensor_core_unsupported_head_size():
    """64-row tiles are built for hk = hv in {128, 256, 512}."""
    w = W.make_workload("wide64", context_lens=[100], num_heads=16, kv_heads=1, head_size_k=64,
                        block_size=16)
    with pytest.raises(pa.PaError) as e:
        run_gpu(w)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


# ---- full-size workloads: sampled sequences ------------------------------------

def sample_rows(w, k, seed):
    rng = np.random.default_rng(seed)
    L = w.context_lens
    pick = {int(np.argmax(L)), int(np.argmin(L))}
    pick |= set(rng.choice(w.batch, size=min(k, w.batch), replace=False).tolist())
    pick = sorted(pick)
    qs = np.concatenate([[0], np.cumsum(w.q_seqlens)])
    rows = np.concatenate([np.arange(qs[b], qs[b + 1]) for b in pick])
    return pick, rows


@pytest.mark.slow
@pytest.mark.parametrize("name", ["gqa_decode", "spec_decode", "alibi_decode", "mqa_split",
                                  "mla_decode", "prefill_causal"])
def test_full_size_sampled(oracle_mod, name):
    w = W.NAMED[name]()
    got, db = run_gpu(w)
    pick, rows = sample_rows(w, {"mqa_split": 2, "prefill_causal": 1}.get(name, 6), 99)
    ref, _ = oracle_mod.attention(w, subset=pick, threads=CORES)
    compare(got, ref, rows)
    # every output row is finite (NaN-poisoned tail slots and spare blocks never read)
    assert np.isfinite(got).all()
