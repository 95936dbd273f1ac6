"""Host-side pieces of the benchmark that run without a GPU: the kernel whose
ncu summary a workload's roofline line cites must be the one pa_forward
dispatches (tile height by the work list's rule), and the step-time
percentiles."""
import numpy as np
import pytest

import bench
import paged_kv_cache_206_gb300 as pa
from paged_kv_cache_206_gb300 import workloads as W

# which kernel each benchmark workload runs, by its tile height and head sizes
EXPECTED = {
    "tiny_decode": "fma_decode_kernel",      # 1 row per (sequence, kv head)
    "gqa_decode": "mma_decode_kernel",       # 4 rows, hk = hv = 128
    "spec_decode": "mma_decode_kernel",      # 4 rows (q = 4)
    "alibi_decode": "fma_decode_kernel",     # 1 row
    "mqa_split": "tc_decode_kernel",         # 64 rows, 512 dims
    "mla_decode": "wide_decode_kernel",      # 16 rows over a shared 576/512 cache
    "prefill_causal": "pf_pair_kernel",      # 2048 rows -> 256-row tiles
}


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_206_gb300 import build_lib
    build_lib.build()
    return pa.load_library()


def _light(name):
    """The workload's configuration without filling its caches."""
    rows = {"tiny_decode": (4, 4, 64, 64, 1), "gqa_decode": (32, 8, 128, 128, 1),
            "spec_decode": (32, 32, 128, 128, 4), "alibi_decode": (40, 40, 128, 128, 1),
            "mqa_split": (64, 1, 512, 512, 1), "mla_decode": (16, 1, 576, 512, 1),
            "prefill_causal": (32, 32, 128, 128, 2048)}[name]
    H, Hk, hk, hv, q = rows
    return pa.make_config(batch=2, num_heads=H, kv_heads=Hk, head_size_k=hk, head_size_v=hv,
                          block_size=64, num_blocks=100, max_blocks_per_seq=40, max_seqlen_q=q,
                          num_sms=152)


@pytest.mark.parametrize("name", sorted(EXPECTED))
def test_dominant_kernel_matches_dispatch(lib, name):
    cfg = _light(name)
    assert bench.dominant_kernel(cfg, name == "mla_decode") == EXPECTED[name]
    # the tile height the planner uses agrees with that kernel's row range
    L = 2048 if cfg.max_seqlen_q > 1 else 300
    ql = np.array([cfg.max_seqlen_q] * 2, np.int32) if cfg.max_seqlen_q > 1 else None
    p = pa.pa_plan(cfg, np.array([L, L], np.int32), ql)
    tile = int((p.work[:, 3] - p.work[:, 2]).max())
    rows = (cfg.num_heads // cfg.kv_heads) * cfg.max_seqlen_q
    want = {"fma_decode_kernel": rows, "mma_decode_kernel": rows, "tc_decode_kernel": min(64, rows),
            "wide_decode_kernel": rows,
            "pf_attn_kernel": 128, "pf_pair_kernel": 256}[EXPECTED[name]]
    assert tile == want
    # every kernel named has its device sources listed for the profile check
    assert EXPECTED[name] in bench.KERNEL_SOURCES


def test_named_workloads_are_covered():
    assert set(EXPECTED) == set(W.NAMED)


def test_percentiles_nearest_rank():
    xs = list(range(1, 12))  # 1..11
    p = bench.percentiles(xs)
    assert p == {"median": 6, "p10": 2, "p90": 10}
    assert bench.percentiles([5.0]) == {"median": 5.0, "p10": 5.0, "p90": 5.0}


@pytest.mark.parametrize("make", [
    lambda: W.tiny_decode(seed=3),
    lambda: W.make_workload("spec", context_lens=[40, 300, 90], q_seqlens=[2, 4, 3], num_heads=8,
                            kv_heads=4, head_size_k=64, block_size=16,
                            mask_type=W.MASK_NORM_COMPRESS, seed=4),
    lambda: W.make_workload("alibi", context_lens=[70, 20], num_heads=6, kv_heads=3,
                            head_size_k=64, block_size=16, mask_type=W.MASK_ALIBI, seed=5),
    lambda: W.make_workload("shared", context_lens=[50, 33, 80], num_heads=8, kv_heads=2,
                            head_size_k=128, head_size_v=64, block_size=16, seed=6,
                            shared_kv=True),
])
def test_reference_sample_is_a_slice_of_the_workload(oracle_mod, make):
    """The reference arm's per-step sample (first sequences x first kv heads)
    is the same attention problem restricted: the oracle on it equals the
    matching rows and heads of the oracle on the whole batch."""
    w = make()
    full, _ = oracle_mod.attention(w, threads=2)
    G = w.num_heads // w.kv_heads
    for nseq, nkv in ((1, 1), (w.batch, 1), (w.batch - 1, w.kv_heads)):
        smp = bench.reference_sample(w, nseq, nkv)
        got, _ = oracle_mod.attention(smp, threads=2)
        nq = int(w.q_seqlens[:nseq].sum())
        assert np.array_equal(got, full[:nq, :nkv * G])
        per = w.head_size_k + (0 if w.shared_kv else w.head_size_v)
        assert smp.kv_bytes() == int(w.context_lens[:nseq].sum()) * nkv * per * 2
