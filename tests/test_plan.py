"""Host planner (pa_plan) against the oracle's planner and the constraints.

pa_plan lives in libpa.so but is pure host code, so these run without a GPU.
The work list must equal the oracle's restatement of the rule bit for bit, and
must partition every sequence's KV blocks exactly once per (kv head, tile).
"""
import math

import numpy as np
import pytest

import paged_kv_cache_206_gb300 as pa


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_206_gb300 import build_lib
    build_lib.build()
    return pa.load_library()


def cfg(**kw):
    base = dict(batch=4, num_heads=8, kv_heads=2, head_size_k=128, block_size=16,
                num_blocks=10_000, max_blocks_per_seq=600, max_seqlen_q=1, num_sms=152)
    base.update(kw)
    return pa.make_config(**base)


def oracle_plan(oracle_mod, c, ctx, ql):
    return oracle_mod.plan(c.batch, c.num_heads, c.kv_heads, c.head_size_k, c.head_size_v,
                           c.block_size, c.max_seqlen_q, c.chunk_blocks, c.num_sms, ctx, ql)


def check_partition(c, ctx, ql, plan):
    """Every (b, kvh) has its rows tiled and, per tile, its blocks covered once."""
    G = c.num_heads // c.kv_heads
    seen = {}
    qs = np.concatenate([[0], np.cumsum(ql if ql is not None else np.ones(c.batch, int))])
    for it in plan.work:
        b, kvh, r0, r1, kb0, kb1, q_start, slot = map(int, it)
        assert q_start == qs[b]
        assert 0 <= kb0 < kb1 <= math.ceil(ctx[b] / c.block_size)
        assert 0 <= r0 < r1
        seen.setdefault((b, kvh, r0, r1), []).append((kb0, kb1))
    for b in range(c.batch):
        q = 1 if ql is None else int(ql[b])
        nb = math.ceil(ctx[b] / c.block_size)
        for kvh in range(c.kv_heads):
            tiles = sorted(k[2:] for k in seen if k[0] == b and k[1] == kvh)
            rows = [r for t in tiles for r in range(*t)]
            assert rows == list(range(G * q))
            for t in tiles:
                ranges = sorted(seen[(b, kvh) + t])
                assert ranges[0][0] == 0 and ranges[-1][1] == nb
                assert all(x[1] == y[0] for x, y in zip(ranges, ranges[1:]))


@pytest.mark.parametrize("seed", range(12))
def test_plan_matches_oracle_plan(lib, oracle_mod, seed):
    rng = np.random.default_rng(seed)
    H = int(rng.choice([1, 4, 8, 32, 64]))
    Hk = int(rng.choice([d for d in (1, 2, 4, 8, 32, 64) if H % d == 0]))
    bs = int(rng.choice([16, 32, 128]))
    maxq = int(rng.choice([1, 1, 2, 4, 7]))
    B = int(rng.integers(1, 70))
    ctx = rng.integers(1, 3000, size=B).astype(np.int32)
    ql = None if maxq == 1 else rng.integers(1, maxq + 1, size=B).astype(np.int32)
    if ql is not None:
        ctx = np.maximum(ctx, ql)
    chunk = int(rng.choice([0, 0, 1, 3, 16]))
    hk = int(rng.choice([64, 128, 256]))
    hv = int(rng.choice([hk, 64]))
    c = cfg(batch=B, num_heads=H, kv_heads=Hk, block_size=bs, max_seqlen_q=maxq,
            chunk_blocks=chunk, head_size_k=hk, head_size_v=hv,
            max_blocks_per_seq=int(math.ceil(ctx.max() / bs)),
            num_sms=int(rng.choice([1, 148, 152])))
    plan = pa.pa_plan(c, ctx, ql)
    work, comb, prows = oracle_plan(oracle_mod, c, ctx, ql)
    assert np.array_equal(plan.work, work)
    assert np.array_equal(plan.combine, comb)
    check_partition(c, ctx, ql, plan)
    # workspace: status area, then P*hv fp16 partials, then P fp32 lse, 256-aligned parts
    up = lambda x: (x + 255) // 256 * 256
    assert plan.workspace_bytes == up(up(256 + prows * hv * 2) + prows * 4)


def test_named_workload_plans(lib, oracle_mod):
    """The five named shapes plan as expected (items, splits, combines)."""
    # long-context MQA: 8 seqs x 256 blocks, 16-block chunks -> 128 items, 8 combines
    c = cfg(batch=8, num_heads=64, kv_heads=1, head_size_k=512, block_size=128,
            max_blocks_per_seq=256, chunk_blocks=16)
    p = pa.pa_plan(c, np.full(8, 32768, np.int32))
    assert p.work.shape == (128, 8) and p.combine.shape == (8, 4)
    assert (p.work[:, 2] == 0).all() and (p.work[:, 3] == 64).all()
    assert (p.combine[:, 3] == 16).all()
    # tiny decode, auto chunk c = max(1, ceil(40/1216), ceil(64*1*64/(16*128))) = 2:
    # NB = {3, 7} -> S = {2, 4}; 4 kv heads -> 24 items, 8 combines
    c = cfg(batch=2, num_heads=4, kv_heads=4, head_size_k=64, block_size=16, num_blocks=32,
            max_blocks_per_seq=7, chunk_blocks=0)
    p = pa.pa_plan(c, np.array([37, 100], np.int32))
    assert p.work.shape[0] == 24 and p.combine.shape[0] == 8
    # with one chunk covering everything there is no split and no combine
    c.chunk_blocks = 7
    p = pa.pa_plan(c, np.array([37, 100], np.int32))
    assert p.combine.shape[0] == 0 and (p.work[:, 7] == -1).all()
    assert p.work.shape[0] == 8


def test_auto_chunk_rule_values(lib):
    # c_min dominates for wide tiles: TR=64, hv=512, bs=128, hk+hv=1024 -> 16
    c = cfg(batch=8, num_heads=64, kv_heads=1, head_size_k=512, block_size=128,
            max_blocks_per_seq=256, num_sms=152)
    p = pa.pa_plan(c, np.full(8, 32768, np.int32))
    assert set((p.work[:, 5] - p.work[:, 4]).tolist()) == {16}
    # c_bal dominates for GQA decode: W = sum NB * Hk = 64*32*8 = 16384 -> ceil(16384/1216) = 14
    c = cfg(batch=64, num_heads=32, kv_heads=8, head_size_k=128, block_size=128,
            max_blocks_per_seq=32, num_sms=152)
    p = pa.pa_plan(c, np.full(64, 4096, np.int32))
    assert sorted(set((p.work[:, 5] - p.work[:, 4]).tolist())) == [4, 14]
    # c_min counts the rows a tile really holds: 16 heads on one kv head fill
    # 16 of the 64 rows -> ceil(64*16*512 / (64*(576+512))) = ceil(7.53) = 8
    c = cfg(batch=8, num_heads=16, kv_heads=1, head_size_k=576, head_size_v=512,
            block_size=64, max_blocks_per_seq=128, num_sms=152)
    p = pa.pa_plan(c, np.full(8, 8192, np.int32))
    assert set((p.work[:, 5] - p.work[:, 4]).tolist()) == {8}


def test_tile_height_rule(lib, oracle_mod):
    """Row tiles by the group rows G * max_q and the head sizes: every row of
    a (sequence, kv head) up to 8 rows; 64-row tiles; for hk = hv in {64, 128}
    128-row tiles past 64 rows and 256-row tiles past 128."""
    cases = [  # (heads, kv heads, hk, hv, max_q) -> expected tile height
        ((8, 1, 128, 128, 1), 8), ((16, 1, 128, 128, 1), 64), ((16, 1, 128, 128, 4), 64),
        ((16, 1, 128, 128, 5), 128), ((32, 1, 128, 128, 4), 128), ((1, 1, 64, 64, 128), 128),
        ((1, 1, 64, 64, 129), 256), ((32, 1, 128, 128, 5), 256), ((64, 1, 512, 512, 1), 64),
        ((16, 1, 256, 256, 9), 64), ((16, 1, 576, 512, 9), 64), ((2, 1, 128, 128, 300), 256),
    ]
    for (H, Hk, hk, hv, q), tr in cases:
        c = cfg(batch=1, num_heads=H, kv_heads=Hk, head_size_k=hk, head_size_v=hv,
                block_size=64, max_seqlen_q=q, max_blocks_per_seq=40, chunk_blocks=100)
        rows = (H // Hk) * q
        ql = np.array([q], np.int32) if q > 1 else None
        p = pa.pa_plan(c, np.array([max(q, 300)], np.int32), ql)
        got = int(p.work[0, 3] - p.work[0, 2])
        assert got == min(tr, rows), ((H, Hk, hk, hv, q), got, tr)
        assert p.work.shape[0] == -(-rows // tr)
        work, _, _ = oracle_plan(oracle_mod, c, np.array([max(q, 300)], np.int32), ql)
        assert np.array_equal(work, p.work)
        assert pa.list_capacity(c)[1] == -(-rows // tr)


def test_auto_chunk_wave_fit(lib, oracle_mod):
    """Row tiles above 8 rows run one CTA per SM, so the automatic chunk is
    then refined: of c0 .. min(2 c0, c0 + 31, max(c0, max NB)) the chunk with
    the least ceil(items / num_sms) * chunk is taken, the first on a tie."""
    # 16 heads on one kv head (TR = 64, 16 real rows), hk = hv = 128, bs = 128,
    # 4 SMs: c_min = ceil(64*16*128 / (128*256)) = 4.
    base = dict(num_heads=16, kv_heads=1, head_size_k=128, block_size=128, num_sms=4,
                max_blocks_per_seq=20)
    # six sequences of 20 blocks: c_bal = ceil(120 / 8) = 15 gives 12 items in
    # 3 waves (cost 45); chunks 16-19 keep 12 items (48..57); 20 gives 6 items
    # in 2 waves (cost 40), and the search stops at max NB = 20
    c = cfg(batch=6, **base)
    ctx = np.full(6, 20 * 128, np.int32)
    p = pa.pa_plan(c, ctx)
    assert p.work.shape[0] == 6 and p.combine.shape[0] == 0
    assert set((p.work[:, 5] - p.work[:, 4]).tolist()) == {20}
    # one sequence of 9 blocks: W = 109, c_bal = 14: 11 items, 3 waves (42);
    # 15..19: 11 items (45..57); 20: 6 items, 2 waves (40)
    ctx = np.array([20 * 128] * 5 + [9 * 128], np.int32)
    p = pa.pa_plan(c, ctx)
    assert p.work.shape[0] == 6
    assert sorted(set((p.work[:, 5] - p.work[:, 4]).tolist())) == [9, 20]
    # three sequences of 20 blocks: c_bal = ceil(60/8) = 8 gives 9 items in 3
    # waves (24); 9 keeps 9 items (27); 10 gives 6 items in 2 waves (20), and
    # nothing up to 16 is cheaper
    c = cfg(batch=3, **base)
    p = pa.pa_plan(c, np.full(3, 20 * 128, np.int32))
    assert p.work.shape[0] == 6 and set((p.work[:, 5] - p.work[:, 4]).tolist()) == {10}
    # already a single wave at c0 (one sequence of 20 blocks on 8 SMs:
    # c0 = max(ceil(20/16), 4) = 4, 5 items): a longer chunk only costs
    c = cfg(batch=1, **dict(base, num_sms=8))
    p = pa.pa_plan(c, np.full(1, 20 * 128, np.int32))
    assert p.work.shape[0] == 5 and set((p.work[:, 5] - p.work[:, 4]).tolist()) == {4}
    # the same configurations through the oracle's restatement of the rule
    for b, ctx in ((6, np.full(6, 2560, np.int32)),
                   (6, np.array([2560] * 5 + [1152], np.int32)), (3, np.full(3, 2560, np.int32))):
        cc = cfg(batch=b, **base)
        work, comb, _ = oracle_plan(oracle_mod, cc, ctx, None)
        hp = pa.pa_plan(cc, ctx)
        assert np.array_equal(work, hp.work) and np.array_equal(comb, hp.combine)


@pytest.mark.parametrize("seed", range(12))
def test_wave_fit_matches_oracle_with_few_sms(lib, oracle_mod, seed):
    """Wide tiles on few SMs, where the wave fit moves the chunk most often:
    pa_plan equals the oracle's planner bit for bit."""
    rng = np.random.default_rng(700 + seed)
    G = int(rng.choice([16, 32, 64]))
    Hk = int(rng.choice([1, 2]))
    hk = int(rng.choice([64, 128, 576]))
    hv = 512 if hk == 576 else hk
    bs = int(rng.choice([16, 64, 128]))
    maxq = int(rng.choice([1, 1, 3]))
    B = int(rng.integers(1, 60))
    ctx = rng.integers(1, 6000, size=B).astype(np.int32)
    ql = None if maxq == 1 else rng.integers(1, maxq + 1, size=B).astype(np.int32)
    if ql is not None:
        ctx = np.maximum(ctx, ql)
    c = cfg(batch=B, num_heads=G * Hk, kv_heads=Hk, head_size_k=hk, head_size_v=hv,
            block_size=bs, max_seqlen_q=maxq, max_blocks_per_seq=int(-(-ctx.max() // bs)),
            chunk_blocks=0, num_sms=int(rng.choice([1, 3, 7, 16, 152])))
    hp = pa.pa_plan(c, ctx, ql)
    work, comb, _ = oracle_plan(oracle_mod, c, ctx, ql)
    assert np.array_equal(work, hp.work) and np.array_equal(comb, hp.combine)
    check_partition(c, ctx, ql, hp)


def test_two_call_convention_and_small_buffers(lib):
    import ctypes
    c = cfg(batch=3, chunk_blocks=2)
    ctx = np.array([100, 5, 64], np.int32)
    n, m, ws = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
    assert lib.pa_plan(ctypes.byref(c), ctx.ctypes.data_as(ctypes.c_void_p), None, None, 0,
                       ctypes.byref(n), None, 0, ctypes.byref(m), ctypes.byref(ws)) == pa.PA_OK
    assert n.value > 0 and m.value > 0 and ws.value > 256
    small = np.zeros((n.value - 1) * 8, np.int32)
    st = lib.pa_plan(ctypes.byref(c), ctx.ctypes.data_as(ctypes.c_void_p), None,
                     small.ctypes.data_as(ctypes.c_void_p), n.value - 1, ctypes.byref(n), None, 0,
                     ctypes.byref(m), ctypes.byref(ws))
    assert st == pa.PA_ERR_BUFFER_TOO_SMALL
    assert not small.any()


def status_of(c, ctx, ql=None):
    try:
        pa.pa_plan(c, np.asarray(ctx, np.int32), None if ql is None else np.asarray(ql, np.int32))
    except pa.PaError as e:
        return e.status
    return pa.PA_OK


@pytest.mark.parametrize("kw,ctx,ql,expect", [
    (dict(block_size=24), [10], None, pa.PA_ERR_INVALID_ARG),           # block_size % 16
    (dict(block_size=0), [10], None, pa.PA_ERR_INVALID_ARG),
    (dict(batch=2049), [1] * 2049, None, pa.PA_ERR_INVALID_ARG),       # batch <= 2048
    (dict(batch=0), [], None, pa.PA_ERR_INVALID_ARG),
    (dict(num_heads=6, kv_heads=4), [10] * 4, None, pa.PA_ERR_INVALID_ARG),  # GQA divisibility
    (dict(head_size_k=592), [10] * 4, None, pa.PA_ERR_INVALID_ARG),    # head size <= 576
    (dict(head_size_k=72), [10] * 4, None, pa.PA_ERR_INVALID_ARG),     # multiple of 16
    (dict(head_size_k=320, block_size=256), [10] * 4, None, pa.PA_ERR_INVALID_ARG),
    (dict(max_seqlen_q=2, block_size=256), [10] * 4, [2] * 4, pa.PA_ERR_INVALID_ARG),
    (dict(max_seqlen_q=4), [3, 10, 10, 10], [4, 1, 1, 1], pa.PA_ERR_INVALID_ARG),  # L >= q
    (dict(max_seqlen_q=2), [10] * 4, [3, 1, 1, 1], pa.PA_ERR_INVALID_ARG),         # q <= max
    (dict(), [0, 1, 1, 1], None, pa.PA_ERR_INVALID_ARG),               # L >= 1
    (dict(max_blocks_per_seq=2), [33, 1, 1, 1], None, pa.PA_ERR_INVALID_ARG),  # table too narrow
    (dict(mask_type=4), [10] * 4, None, pa.PA_ERR_UNSUPPORTED),        # spec mask: unspecified
    (dict(mask_type=3), [10] * 4, None, pa.PA_ERR_INVALID_ARG),
    (dict(mask_type=5, max_seqlen_q=2049, block_size=16), [3000] * 4, [2049] * 4,
     pa.PA_ERR_INVALID_ARG),
    (dict(chunk_blocks=0, num_sms=0), [10] * 4, None, pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), [10] * 4, None, pa.PA_ERR_INVALID_ARG),
    (dict(), [10, 20, 30, 40], None, pa.PA_OK),
    (dict(max_blocks_per_seq=3), [33, 1, 1, 48], None, pa.PA_OK),
])
def test_constraint_errors(lib, kw, ctx, ql, expect):
    kw = dict(kw)
    kw.setdefault("batch", len(ctx))
    assert status_of(cfg(**kw), ctx, ql) == expect


@pytest.mark.parametrize("seed", range(10))
def test_list_capacity_bounds_every_plan(lib, seed):
    """pa.list_capacity, the list sizes HostStep reserves, bounds the lists of
    any lengths the configuration admits: all full, all one block, a mix, and
    lengths just past a chunk boundary (the worst case for ceil(NB / c))."""
    rng = np.random.default_rng(100 + seed)
    H = int(rng.choice([4, 8, 32, 64]))
    Hk = int(rng.choice([d for d in (1, 2, 4, 8) if H % d == 0]))
    bs = int(rng.choice([16, 32, 128]))
    maxq = int(rng.choice([1, 2, 4, 9]))
    B = int(rng.integers(1, 200))
    maxnb = int(rng.integers(1, 300))
    chunk = int(rng.choice([0, 0, 1, 5]))
    c = cfg(batch=B, num_heads=H, kv_heads=Hk, block_size=bs, max_seqlen_q=maxq,
            chunk_blocks=chunk, max_blocks_per_seq=maxnb, num_sms=int(rng.choice([1, 152])))
    wcap, ccap = pa.list_capacity(c)
    ql = None if maxq == 1 else np.full(B, maxq, np.int32)
    floor = maxq if ql is not None else 1
    trials = [np.full(B, maxnb * bs), np.full(B, 1), rng.integers(1, maxnb * bs + 1, size=B)]
    n = pa.pa_plan(c, np.maximum(trials[0], floor).astype(np.int32), ql)
    # lengths with NB = k*c + 1 for the chunk the full plan chose
    cc = max(1, int(n.work[0, 5] - n.work[0, 4]))
    nb = np.minimum(maxnb, (rng.integers(0, maxnb // cc + 1, size=B) * cc + 1))
    trials.append(nb * bs - bs + 1)
    for ctx in trials:
        p = pa.pa_plan(c, np.maximum(ctx, floor).astype(np.int32), ql)
        assert p.work.shape[0] <= wcap
        assert p.combine.shape[0] <= ccap
