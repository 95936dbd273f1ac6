"""Seeded random shapes against the oracle.

Each case is drawn from one kernel family (the CUDA-core and warp-MMA decode
kernels for up to 8 rows per kv head, the 16-row shared-KV kernel, the tcgen05
decode kernel for up to 64 rows, the prefill kernels beyond 64) with its
head sizes, block size, query lengths, mask, cache layout and chunking drawn
at random within the limits of pa.h, and compared element by element with the
fp64 oracle. The CPU test checks that every drawn case plans and that the
draw covers every family and option; the GPU test runs them.
"""
import numpy as np
import pytest

import paged_kv_cache_206_gb300 as pa
from paged_kv_cache_206_gb300 import build_lib
from paged_kv_cache_206_gb300 import workloads as W

N_CASES = 36
SEED = 2026


def _family(G, maxq, hk, hv, shared):
    rows = G * maxq
    if rows <= 8:
        return "warp"
    if rows > 64 and hk == hv and hk in (64, 128):
        return "prefill"
    if rows <= 16 and shared and ((hk, hv) == (576, 512) or (hk == hv and hk in (256, 512))):
        return "wide"
    return "tc"


def draw(i):
    """Keyword arguments of workloads.make_workload for case i, and its family."""
    rng = np.random.default_rng([SEED, i])
    fam = ["warp", "warp", "tc", "wide", "prefill"][i % 5]
    shared = False
    if fam == "warp":
        G = int(rng.choice([1, 2, 4, 8]))
        q = int(rng.choice([1, 1, 2])) if G <= 4 else 1
        if G * q > 8:
            q = 1
        hk, hv = [(64, 64), (80, 48), (96, 96), (128, 128), (192, 192), (256, 256), (512, 512),
                  (576, 512)][int(rng.integers(0, 8))]
        shared = hv <= hk and bool(rng.random() < 0.3)
    elif fam == "tc":
        G, q = [(16, 1), (24, 1), (32, 1), (64, 1), (16, 2), (8, 4), (12, 3)][int(rng.integers(0, 7))]
        hk, hv = [(128, 128), (256, 256), (512, 512), (576, 512)][int(rng.integers(0, 4))]
        shared = bool(rng.random() < 0.3) and G * q > 16  # 16-row shared caches go to the wide kernel
    elif fam == "wide":
        G, q = [(16, 1), (12, 1), (8, 2), (10, 1)][int(rng.integers(0, 4))]
        hk, hv = [(576, 512), (256, 256), (512, 512)][int(rng.integers(0, 3))]
        shared = True
    else:
        G = int(rng.choice([1, 2, 4]))
        hk = hv = int(rng.choice([64, 128]))
        q = int(rng.integers(70, 200)) if G == 1 else int(rng.integers(20, 90))
        if G * q <= 64:
            q = 65 // G + 1
    kv_heads = int(rng.choice([1, 2]))
    bs_choices = [16, 32, 48, 64, 128] if (q == 1 and max(hk, hv) <= 256) else [16, 32, 64, 128]
    bs = int(rng.choice(bs_choices))
    B = int(rng.integers(2, 4))
    lens = [int(rng.integers(q, q + 600)) for _ in range(B)]
    if fam == "prefill" and rng.random() < 0.5:
        lens = [q] * B  # q = L: PA_ENCODER-style prefill
    masks = [W.MASK_NONE, W.MASK_ALIBI, W.MASK_NORM_COMPRESS, W.MASK_NORM]
    mask = int(masks[int(rng.integers(0, 4))])
    chunk = int(rng.choice([0, 0, 1, 2, 5]))
    kw = dict(context_lens=lens, q_seqlens=q, num_heads=G * kv_heads, kv_heads=kv_heads,
              head_size_k=hk, head_size_v=hv, block_size=bs, mask_type=mask,
              seed=1000 + i, chunk_blocks=chunk, shared_kv=shared,
              std=0.5 if max(hk, hv) >= 256 else 1.0)
    assert _family(G, q, hk, hv, shared) == fam, (i, fam, G, q, hk, hv, shared)
    return kw, fam


def make(i):
    kw, _ = draw(i)
    return W.make_workload(f"rand{i}", **kw)


# A wider draw: any head sizes the kernels take (multiples of 16 up to 576, K
# and V apart for up to 8 rows a kv head), block sizes 16-256, batches of 1-4,
# lengths on and around block boundaries and past the 2048 of the compressed
# mask, extra block-table columns.
N_WIDE = 160
TC_HEADS = [(128, 128), (256, 256), (512, 512), (576, 512)]


def _supported(rows, hk, hv):
    if rows <= 8:
        return True
    if rows > 64 and hk == hv and hk in (64, 128):
        return True
    return (hk, hv) in TC_HEADS


def draw_wide(i):
    rng = np.random.default_rng([SEED + 1, i])
    while True:
        kind = int(rng.integers(0, 4))
        if kind == 0:      # up to 8 rows a kv head: any head sizes
            G = int(rng.choice([1, 2, 3, 4, 5, 8]))
            q = int(rng.choice([1, 1, 1, 2])) if G <= 4 else 1
            if G >= 2 and rng.random() < 0.3:  # the warp-MMA kernel's head sizes
                hk, hv = [(64, 64), (128, 128), (256, 256), (512, 512), (576, 512)][int(rng.integers(0, 5))]
            else:
                hk = 16 * int(rng.integers(1, 37))
                hv = 16 * int(rng.integers(1, 37)) if rng.random() < 0.4 else hk
        elif kind == 1:    # 9-64 rows: the tensor-core head sizes
            G, q = [(9, 1), (16, 1), (17, 1), (24, 1), (33, 1), (48, 1), (64, 1), (5, 2), (16, 3),
                    (8, 8), (21, 3)][int(rng.integers(0, 11))]
            hk, hv = TC_HEADS[int(rng.integers(0, 4))]
        elif kind == 2:    # prefill-like: more than 64 rows
            G = int(rng.choice([1, 2, 4, 8]))
            q = int(rng.integers(65 // G + 1, 65 // G + 120))
            hk = hv = int(rng.choice([64, 128, 128, 256, 512]))
        else:              # 9-16 rows over a shared cache
            G, q = [(9, 1), (16, 1), (8, 2), (5, 3)][int(rng.integers(0, 4))]
            hk, hv = [(576, 512), (256, 256), (512, 512), (128, 128)][int(rng.integers(0, 4))]
        rows = G * q
        if max(hk, hv) > PA_MAX_HEAD or not _supported(rows, hk, hv):
            continue
        shared = hv <= hk and (kind == 3 or bool(rng.random() < 0.25))
        big = max(hk, hv) > 256 or q > 1
        bs = int(rng.choice([16, 32, 48, 64, 80, 112, 128] + ([] if big else [144, 256])))
        B = int(rng.integers(1, 5))
        lens = []
        for _ in range(B):
            r = rng.random()
            if r < 0.2:
                L = q  # only the query tokens
            elif r < 0.4:
                L = max(q, bs * int(rng.integers(1, 6)) + int(rng.integers(-1, 2)))  # around a block edge
            elif r < 0.47 and q <= 8:
                L = int(rng.integers(2049, 2300))  # past the compressed mask's 2048
            else:
                L = int(rng.integers(q, q + 700))
            lens.append(max(L, q))
        masks = [W.MASK_NONE, W.MASK_ALIBI, W.MASK_NORM_COMPRESS, W.MASK_NORM]
        mask = int(masks[int(rng.integers(0, 4))])
        kw = dict(context_lens=lens, q_seqlens=q, num_heads=G * int(rng.choice([1, 2])),
                  head_size_k=hk, head_size_v=hv, block_size=bs, mask_type=mask,
                  seed=5000 + i, chunk_blocks=int(rng.choice([0, 0, 1, 2, 3, 7])),
                  shared_kv=shared, extra_table_cols=int(rng.choice([0, 0, 3])),
                  std=0.5 if max(hk, hv) >= 256 else 1.0)
        kw["kv_heads"] = kw["num_heads"] // G
        return kw


PA_MAX_HEAD = 576


def test_wide_random_cases_plan(lib):
    """Every case of the wider draw is valid for pa_plan."""
    for i in range(N_WIDE):
        w = W.make_workload(f"wide{i}", **draw_wide(i))
        cfg = pa.config_for(w, num_sms=152)
        ql = None if np.all(w.q_seqlens == 1) else w.q_seqlens
        pa.pa_plan(cfg, w.context_lens, ql)


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return pa.load_library()


def test_random_cases_plan_and_cover(lib):
    """Every drawn case is valid for pa_plan, and the draw spans every kernel
    family, mask type, shared and separate caches, splits and no splits."""
    fams, masks, shared, split, unsplit = set(), set(), set(), False, False
    for i in range(N_CASES):
        kw, fam = draw(i)
        w = W.make_workload(f"rand{i}", **kw)
        cfg = pa.config_for(w, num_sms=152)
        ql = None if np.all(w.q_seqlens == 1) else w.q_seqlens
        plan = pa.pa_plan(cfg, w.context_lens, ql)
        fams.add(fam)
        masks.add(kw["mask_type"])
        shared.add(kw["shared_kv"])
        split |= plan.combine.shape[0] > 0
        unsplit |= plan.combine.shape[0] == 0
    assert fams == {"warp", "tc", "wide", "prefill"}
    assert masks == {W.MASK_NONE, W.MASK_ALIBI, W.MASK_NORM_COMPRESS, W.MASK_NORM}
    assert shared == {True, False} and split and unsplit


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_parity(lib, oracle_mod, i):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests.test_gpu_parity import full_parity
    full_parity(oracle_mod, make(i))


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(N_WIDE))
def test_wide_random_case_parity(lib, oracle_mod, i):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests.test_gpu_parity import full_parity
    full_parity(oracle_mod, W.make_workload(f"wide{i}", **draw_wide(i)))


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(24))
def test_planned_paths_agree_bit_for_bit(lib, i):
    """The device planner's step (capacity grids, CTAs past the device counts
    leaving at once) and the recorded graph step (pinned host arena, device
    plan, output straight into pinned memory when small) give the host-planned
    step's output bit for bit: the same lists, the same kernels."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = W.make_workload(f"wide{i}", **draw_wide(i))
    db = pa.DeviceBatch(w)
    host = db.forward().clone().cpu()
    step = pa.DevicePlanStep(db)
    dev = step.run().clone().cpu()
    assert step.status()[0] == pa.PA_OK
    gs = pa.GraphStep(db.cfg, db.key_cache, db.value_cache, w.total_q, mask=db.mask,
                      alibi_slopes=db.alibi_slopes)
    gs.block_tables.copy_(torch.from_numpy(np.ascontiguousarray(w.block_tables)))
    if gs.q_seqlens is not None:
        gs.q_seqlens.copy_(torch.from_numpy(np.ascontiguousarray(w.q_seqlens)))
    gs.context_lens.copy_(torch.from_numpy(np.ascontiguousarray(w.context_lens)))
    gs.query.copy_(torch.from_numpy(np.ascontiguousarray(w.query)))
    graph = gs.run().clone()
    assert gs.status()[0] == pa.PA_OK
    assert torch.equal(host, dev) and torch.equal(host, graph)
