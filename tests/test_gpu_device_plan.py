"""The device planner (pa_plan_device) and the forward pass over its lists.

The device lists must equal pa_plan's bit for bit (the host planner is itself
pinned to the oracle's restatement of the rule in tests/test_plan.py); a
length that breaks a constraint or a capacity that is too small must be
reported through the counts and the status word, with nothing run. A step
recorded once as a CUDA graph (plan + attention + combine) and replayed after
the lengths change in place must match the oracle on each step's lengths
(max-abs 1e-2, mean-abs 1e-3).
"""
import dataclasses
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


def device_lists(cfg, ctx, ql, work_cap=None, comb_cap=None):
    wcap, ccap, ws = pa.pa_plan_bounds(cfg)
    wcap = wcap if work_cap is None else work_cap
    ccap = ccap if comb_cap is None else comb_cap
    d_ctx = torch.from_numpy(np.ascontiguousarray(ctx, dtype=np.int32)).cuda()
    d_ql = None if ql is None else torch.from_numpy(np.ascontiguousarray(ql, dtype=np.int32)).cuda()
    work = torch.full((wcap, pa.PA_WORK_INTS), -7, dtype=torch.int32, device="cuda")
    comb = torch.full((max(ccap, 1), pa.PA_COMBINE_INTS), -7, dtype=torch.int32, device="cuda")
    counts = torch.full((pa.PA_PLAN_COUNTS,), -7, dtype=torch.int32, device="cuda")
    ws_t = torch.zeros(pa.PA_STATUS_BYTES, dtype=torch.uint8, device="cuda")
    lib = pa.load_library()
    import ctypes
    st = lib.pa_plan_device(ctypes.byref(cfg), ctypes.c_void_p(d_ctx.data_ptr()),
                            None if d_ql is None else ctypes.c_void_p(d_ql.data_ptr()),
                            ctypes.c_void_p(work.data_ptr()), wcap,
                            ctypes.c_void_p(comb.data_ptr()), ccap,
                            ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(ws_t.data_ptr()),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pa.PA_OK
    torch.cuda.synchronize()
    c = counts.cpu().numpy()
    return c, work.cpu().numpy(), comb.cpu().numpy(), pa.pa_status_read(ws_t)


def random_case(seed):
    rng = np.random.default_rng(500 + seed)
    H = int(rng.choice([1, 4, 8, 32, 64]))
    Hk = int(rng.choice([d for d in (1, 2, 4, 8, 32, 64) if H % d == 0]))
    bs = int(rng.choice([16, 32, 128]))
    maxq = int(rng.choice([1, 1, 2, 4, 7, 20]))
    B = int(rng.choice([1, 3, 70, 1000, 2048]))
    ctx = rng.integers(1, 5000, size=B).astype(np.int32)
    ql = None if maxq == 1 else rng.integers(1, maxq + 1, size=B).astype(np.int32)
    if ql is not None:
        ctx = np.maximum(ctx, ql)
    chunk = int(rng.choice([0, 0, 1, 3, 16]))
    hk = int(rng.choice([64, 128, 576]))
    hv = 512 if hk == 576 else hk
    cfg = pa.make_config(batch=B, num_heads=H, kv_heads=Hk, head_size_k=hk, head_size_v=hv,
                         block_size=bs if hk <= 256 else min(bs, 128), num_blocks=10 ** 6,
                         max_blocks_per_seq=int(-(-ctx.max() // bs)) + int(rng.integers(0, 3)),
                         max_seqlen_q=maxq, chunk_blocks=chunk,
                         num_sms=int(rng.choice([1, 4, 16, 148, 152])))
    return cfg, ctx, ql


@pytest.mark.parametrize("seed", range(24))
def test_device_plan_equals_host_plan(seed):
    cfg, ctx, ql = random_case(seed)
    host = pa.pa_plan(cfg, ctx, ql)
    counts, work, comb, (st, bits) = device_lists(cfg, ctx, ql)
    assert st == pa.PA_OK and bits == 0
    n, m = host.work.shape[0], host.combine.shape[0]
    assert counts.tolist()[:2] == [n, m] and counts[3] == 0
    assert np.array_equal(work[:n], host.work)
    assert np.array_equal(comb[:m], host.combine)
    # partial rows: the workspace pa_plan sizes holds exactly counts[2] rows
    up = lambda x: (x + 255) // 256 * 256
    assert host.workspace_bytes == up(up(256 + int(counts[2]) * cfg.head_size_v * 2) +
                                      int(counts[2]) * 4)
    # nothing past the counts was written
    assert (work[n:] == -7).all() and (comb[m:] == -7).all()


@pytest.mark.parametrize("seed", range(8))
def test_device_wave_fit_equals_host(seed):
    """Wide tiles (one CTA per SM) with the automatic chunk: the device
    planner's wave fit (one warp per candidate chunk) picks the host's chunk."""
    rng = np.random.default_rng(900 + seed)
    G = int(rng.choice([16, 64]))
    hk = int(rng.choice([128, 576]))
    hv = 512 if hk == 576 else hk
    bs = int(rng.choice([16, 64]))
    B = int(rng.choice([6, 64, 300]))
    ctx = rng.integers(1, 9000, size=B).astype(np.int32)
    cfg = pa.make_config(batch=B, num_heads=G, kv_heads=1, head_size_k=hk, head_size_v=hv,
                         block_size=bs, num_blocks=10 ** 6,
                         max_blocks_per_seq=int(-(-ctx.max() // bs)), chunk_blocks=0,
                         num_sms=int(rng.choice([3, 16, 152])))
    host = pa.pa_plan(cfg, ctx, None)
    counts, work, comb, (st, bits) = device_lists(cfg, ctx, None)
    assert st == pa.PA_OK and bits == 0
    n, m = host.work.shape[0], host.combine.shape[0]
    assert counts.tolist()[:2] == [n, m]
    assert np.array_equal(work[:n], host.work) and np.array_equal(comb[:m], host.combine)


def test_device_plan_reports_bad_lengths_and_small_capacity():
    cfg = pa.make_config(batch=3, num_heads=8, kv_heads=2, head_size_k=128, block_size=16,
                         num_blocks=1000, max_blocks_per_seq=10, max_seqlen_q=4, num_sms=152)
    ok_ctx, ok_ql = np.array([50, 3, 160], np.int32), np.array([4, 3, 1], np.int32)
    # L < q
    counts, work, _, (st, bits) = device_lists(cfg, np.array([50, 2, 160], np.int32), ok_ql)
    assert counts.tolist() == [0, 0, 0, 1] and bits & 8 and st == pa.PA_ERR_INVALID_ARG
    assert (work == -7).all()
    # a table too narrow for L (NB = 11 > 10)
    counts, _, _, (st, bits) = device_lists(cfg, np.array([50, 3, 161], np.int32), ok_ql)
    assert counts[3] == 1 and st == pa.PA_ERR_INVALID_ARG
    # q above max_seqlen_q
    counts, _, _, (st, _) = device_lists(cfg, ok_ctx, np.array([5, 3, 1], np.int32))
    assert counts[3] == 1 and st == pa.PA_ERR_INVALID_ARG
    # capacity one short
    n = pa.pa_plan(cfg, ok_ctx, ok_ql).work.shape[0]
    counts, _, _, (st, bits) = device_lists(cfg, ok_ctx, ok_ql, work_cap=n - 1)
    assert counts.tolist() == [0, 0, 0, 2] and bits & 4 and st == pa.PA_ERR_BUFFER_TOO_SMALL
    counts, _, _, (st, _) = device_lists(cfg, ok_ctx, ok_ql, work_cap=n)
    assert st == pa.PA_OK and counts[0] == n


CASES = {
    "gqa": lambda: W.gqa_decode(batch=6, max_len=1800, seed=70),
    "spec_mask": lambda: W.spec_decode(batch=3, max_len=2600, seed=71),
    "mqa_tc": lambda: W.make_workload("mqa", context_lens=[1500, 300], num_heads=64, kv_heads=1,
                                      head_size_k=512, block_size=64, std=0.5, seed=72),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_graph_replay_with_changing_lengths(oracle_mod, name):
    w = CASES[name]()
    db = pa.DeviceBatch(w)
    step = pa.DevicePlanStep(db)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step.run(s)  # first call: attributes and tensor maps set up outside the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step.run(s)
    q = w.q_seqlens
    for cut in (0, 150, 600):
        lens = np.maximum(w.context_lens - cut, q).astype(np.int32)
        db.context_lens.copy_(torch.from_numpy(lens))
        step.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        st, bits = step.status()
        assert st == pa.PA_OK, (st, bits)
        got = step.out.double().cpu().numpy()
        ref, _ = oracle_mod.attention(dataclasses.replace(w, context_lens=lens), threads=CORES)
        err = np.abs(got - ref)
        assert np.isfinite(got).all()
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (cut, err.max(), err.mean())


@pytest.mark.parametrize("name", sorted(CASES))
def test_graph_step_host_buffers(oracle_mod, name):
    """GraphStep: inputs written into pinned host views, one graph replay per
    step (copy in, device plan, attention, combine, copy out). New lengths and
    a new query between replays must give the oracle's answer for each."""
    w = CASES[name]()
    db = pa.DeviceBatch(w)
    gs = pa.GraphStep(db.cfg, db.key_cache, db.value_cache, w.total_q, mask=db.mask,
                      alibi_slopes=db.alibi_slopes)
    gs.block_tables.copy_(torch.from_numpy(np.ascontiguousarray(w.block_tables)))
    if gs.q_seqlens is not None:
        gs.q_seqlens.copy_(torch.from_numpy(np.ascontiguousarray(w.q_seqlens)))
    rng = np.random.default_rng(90)
    q = w.q_seqlens
    for step, cut in enumerate((0, 150, 600)):
        lens = np.maximum(w.context_lens - cut, q).astype(np.int32)
        query = w.query if step == 0 else (
            rng.standard_normal(w.query.shape) * 0.5).astype(np.float16)
        wi = dataclasses.replace(w, context_lens=lens, query=query)
        gs.context_lens.copy_(torch.from_numpy(lens))
        gs.query.copy_(torch.from_numpy(np.ascontiguousarray(query)))
        gs.out.fill_(float("nan"))
        got = gs.run().double().numpy()
        st, bits = gs.status()
        assert st == pa.PA_OK, (st, bits)
        ref, _ = oracle_mod.attention(wi, threads=CORES)
        err = np.abs(got - ref)
        assert np.isfinite(got).all()
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (cut, err.max(), err.mean())
    assert gs.graph is not None
