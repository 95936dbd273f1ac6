"""Failure detection on the GPU without a GPU fault.

Every wait in the decode kernels is bounded: a role that waits for another
role's progress gives up after a cycle limit, sets PA_STATUS_BIT_TIMEOUT, lets
the copies and tensor-core operations it issued finish, frees its tensor
memory and exits. The limit is about two seconds, so a healthy launch never
meets it; the test hook pa_testing_set_wait_limit lowers it to a few dozen
cycles, far below the latency of any copy, so that the waits of a correct
launch run out. The launch must then report PA_ERR_TIMEOUT through the status
word, and the context must stay usable: with the default limit back, the same
batch matches the oracle.
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
    yield
    pa.testing_set_wait_limit(0)


def compare(got, ref):
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())


CASES = {
    # mma.sync kernel (4 rows: GQA 32/8), warp-pipelined TMA ring, split items
    "warp_pipe_gqa": (lambda: W.gqa_decode(batch=8, max_len=3000, seed=60), 2),
    # CUDA-core kernel (1 row), ALiBi
    "warp_pipe_fma": (lambda: W.alibi_decode(batch=16, max_len=2048, seed=61), 3),
    # tcgen05 kernel, 16 rows, 16-token blocks, split items
    "tc_r16_bs16": (lambda: W.make_workload("r16", context_lens=[100, 300, 17, 129],
                                            num_heads=16, kv_heads=1, head_size_k=128,
                                            block_size=16, seed=62), 2),
    # 16-row warp-level MMA kernel, shared 576/512 cache, split items
    "wide_mla": (lambda: W.make_workload("wmla", context_lens=[900, 300, 65], num_heads=16,
                                         kv_heads=1, head_size_k=576, head_size_v=512,
                                         block_size=64, std=0.5, seed=64, shared_kv=True), 4),
    # tcgen05 kernel, 64 rows of a 512-dim MQA head
    "tc_mqa_hd512": (lambda: W.make_workload("mqa", context_lens=[1500, 700], num_heads=64,
                                             kv_heads=1, head_size_k=512, block_size=128,
                                             std=0.5, seed=63), 4),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_short_wait_limit_times_out_and_the_context_survives(oracle_mod, name):
    make, chunk = CASES[name]
    w = make()
    db = pa.DeviceBatch(w, chunk_blocks=chunk)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=db.out.device)
    # Whether a wait outlasts 32 cycles depends on when its copy lands: the
    # L2 is flushed first so that the copies come from HBM, and the launch is
    # tried up to three times; one report of a timeout is what is checked.
    st, bits = pa.PA_OK, 0
    for _ in range(3):
        flush.zero_()
        pa.testing_set_wait_limit(32)
        try:
            db.forward()
            st, bits = db.status()
        finally:
            pa.testing_set_wait_limit(0)
        if st == pa.PA_ERR_TIMEOUT:
            break
        pa.pa_status_clear(db.workspace)
    assert st == pa.PA_ERR_TIMEOUT, (pa.status_string(st), bits)
    assert bits & pa.PA_STATUS_BIT_TIMEOUT
    # the context is still usable: the same batch, with the default limit and a
    # cleared status word, matches the oracle
    torch.cuda.synchronize()
    pa.pa_status_clear(db.workspace)
    got = db.forward().float().cpu().numpy().astype(np.float64)
    st, bits = db.status()
    assert st == pa.PA_OK, (pa.status_string(st), bits)
    ref, _ = oracle_mod.attention(w, threads=CORES)
    compare(got, ref)
