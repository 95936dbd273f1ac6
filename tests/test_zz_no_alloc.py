"""pa_forward_noalloc, the entry point for callers that cannot allocate device
memory (a pool- or runtime-owned memory budget, or a latency-critical loop that
cannot take cudaMalloc's implicit synchronisation): it must give the same
attention as pa_forward with a caller-provided workspace, call after call.

The library's fixed device array keeps the previous call's contents, so the
test runs the entry point twice in a row on split-KV workloads (partial results
go through the array) and compares both outputs with pa_forward, within the
tolerance of the parity tests (max-abs 1e-2, mean-abs 1e-3). This file is named
to run last; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import paged_kv_cache_206_gb300 as pa
from paged_kv_cache_206_gb300 import build_lib
from paged_kv_cache_206_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.build()
    pa.load_library()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(db, out, status, workspace_bytes=None, block_tables=None):
    """The C ABI call itself (through ctypes), on the current stream."""
    lib = pa.load_library()
    n_comb = 0 if db.combine is None else db.combine.shape[0]
    bt = db.block_tables if block_tables is None else block_tables
    return lib.pa_forward_noalloc(
        ctypes.byref(db.cfg), _ptr(db.query), _ptr(db.key_cache), _ptr(db.value_cache),
        _ptr(bt), _ptr(db.context_lens), _ptr(db.q_seqlens), _ptr(db.mask),
        _ptr(db.alibi_slopes), _ptr(db.work), db.work.shape[0], _ptr(db.combine), n_comb,
        db.plan.workspace_bytes if workspace_bytes is None else workspace_bytes, _ptr(status),
        _ptr(out), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = {
    # CUDA-core / mma.sync path with many splits
    "gqa_split": (lambda: W.gqa_decode(batch=6, max_len=1500, seed=40), 2),
    # spec decode with the compressed mask, split
    "spec_split": (lambda: W.spec_decode(batch=3, max_len=2600, seed=41), 3),
    # tcgen05 path: 64-row tiles of a 512-dim MQA head, split
    "mqa_split": (lambda: W.make_workload("mqa", context_lens=[2085, 700], num_heads=64,
                                          kv_heads=1, head_size_k=512, block_size=128,
                                          std=0.5, seed=42), 4),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_pa_forward_twice(name):
    make, chunk = CASES[name]
    w = make()
    db = pa.DeviceBatch(w, chunk_blocks=chunk)
    assert db.combine is not None, "the case must exercise split-KV partials"
    assert db.plan.workspace_bytes <= pa.PA_NOALLOC_SCRATCH_BYTES
    ref = db.forward().clone()
    assert db.status()[0] == pa.PA_OK
    ref64 = ref.double()
    status = torch.zeros(1, dtype=torch.int32, device=db.out.device)
    for _ in range(2):
        out = torch.full_like(db.out, float("nan"))
        status.fill_(-1)
        assert call_noalloc(db, out, status) == pa.PA_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.isfinite(out).all()
        err = (out.double() - ref64).abs()
        assert err.max().item() <= MAX_ABS
        assert err.mean().item() <= MEAN_ABS


def test_noalloc_rejects_workspace_beyond_its_array():
    w = W.gqa_decode(batch=2, max_len=300, seed=43)
    db = pa.DeviceBatch(w, chunk_blocks=1)
    out = torch.empty_like(db.out)
    st = call_noalloc(db, out, None, workspace_bytes=pa.PA_NOALLOC_SCRATCH_BYTES + 1)
    assert st == pa.PA_ERR_BUFFER_TOO_SMALL


def test_noalloc_status_reaches_the_caller_and_is_cleared_per_call():
    """Each call starts from a cleared status word in the shared array, and a
    kernel's status bit reaches the caller's `status`. The fault is made on the
    host: one block-table entry past num_blocks, which the kernel flags and
    never dereferences. The next clean call must report 0 again."""
    w = W.gqa_decode(batch=4, max_len=600, seed=44)
    db = pa.DeviceBatch(w, chunk_blocks=2)
    assert db.combine is not None
    bad = db.block_tables.clone()
    bad[2, 0] = w.num_blocks + 5
    status = torch.zeros(1, dtype=torch.int32, device=db.out.device)
    out = torch.empty_like(db.out)
    assert call_noalloc(db, out, status, block_tables=bad) == pa.PA_OK
    torch.cuda.synchronize()
    assert int(status.item()) & pa.PA_STATUS_BIT_BLOCK_INDEX
    status.fill_(-1)
    assert call_noalloc(db, out, status) == pa.PA_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = db.forward()
    assert db.status()[0] == pa.PA_OK
    err = (out.double() - ref.double()).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
