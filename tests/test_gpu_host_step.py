"""HostStep: the step fed from pinned host buffers (one host-to-device copy of
an arena that pa_plan fills with the work lists) gives the same output, bit
for bit, as the device-resident DeviceBatch run of the same plan, and agrees
with the oracle within the parity tolerance (max-abs 1e-2, mean-abs 1e-3).
It also runs several steps in a row with changing context lengths, which
re-plans into the same arena."""
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


def host_step_for(db, w):
    hs = pa.HostStep(db.cfg, db.key_cache, db.value_cache, w.total_q, mask=db.mask,
                     alibi_slopes=db.alibi_slopes)
    hs.query.copy_(torch.from_numpy(np.ascontiguousarray(w.query)))
    hs.block_tables.copy_(torch.from_numpy(np.ascontiguousarray(w.block_tables)))
    hs.context_lens.copy_(torch.from_numpy(np.ascontiguousarray(w.context_lens)))
    if hs.q_seqlens is not None:
        hs.q_seqlens.copy_(torch.from_numpy(np.ascontiguousarray(w.q_seqlens)))
    return hs


CASES = {
    "gqa_split": lambda: W.gqa_decode(batch=5, max_len=1700, seed=60),
    "spec_mask": lambda: W.spec_decode(batch=3, max_len=2400, seed=61),
    "mqa_tc": lambda: W.make_workload("mqa", context_lens=[900, 2100], num_heads=64, kv_heads=1,
                                      head_size_k=512, block_size=64, std=0.5, seed=62),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_host_step_matches_device_batch_and_oracle(oracle_mod, name):
    w = CASES[name]()
    db = pa.DeviceBatch(w)
    ref_dev = db.forward().cpu()
    hs = host_step_for(db, w)
    out = hs.run()
    assert hs.status()[0] == pa.PA_OK
    assert hs.n_items == db.plan.work.shape[0]
    assert torch.equal(out, ref_dev)
    ref, _ = oracle_mod.attention(w, threads=CORES)
    err = np.abs(out.double().numpy() - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS


def test_host_step_replans_each_step(oracle_mod):
    """Shrinking the context lengths between steps changes the plan; each step
    must match the oracle run on the lengths of that step."""
    w = W.gqa_decode(batch=4, max_len=1500, seed=63)
    db = pa.DeviceBatch(w)
    hs = host_step_for(db, w)
    for cut in (0, 200, 700):
        lens = np.maximum(w.context_lens - cut, 1).astype(np.int32)
        hs.context_lens.copy_(torch.from_numpy(lens))
        out = hs.run().double().numpy()
        assert hs.status()[0] == pa.PA_OK
        w2 = dataclasses.replace(w, context_lens=lens)
        ref, _ = oracle_mod.attention(w2, threads=CORES)
        err = np.abs(out - ref)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS
