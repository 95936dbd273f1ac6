"""CPU oracle for paged attention (double precision).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers. The library's product path never
imports this package, and this package imports nothing from the library.

``build()`` compiles ``pa_oracle.c`` with gcc (OpenMP) into
``oracle/_build/liboracle.so``; ``attention()`` and ``plan()`` call it through
ctypes. See ``pa_oracle.c`` for what each function follows on the pages.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def _stamp() -> str:
    """The machine and compiler the library is built for: one built elsewhere
    is never reused."""
    ver = subprocess.run(["gcc", "--version"], capture_output=True, text=True).stdout
    return platform.machine() + " " + ver.splitlines()[0] if ver else platform.machine()


def build(force: bool = False) -> str:
    """Compile the oracle if its shared library is missing, stale, or built for
    another machine or compiler."""
    stamp_path = _OUT + ".stamp"
    stamp = _stamp()
    same = os.path.exists(stamp_path) and open(stamp_path).read().strip() == stamp
    if (not force and same and os.path.exists(_OUT)
            and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC)):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC,
                    "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _OUT)
    with open(stamp_path, "w") as f:
        f.write(stamp + "\n")
    return _OUT


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_attention.restype = i32
        lib.oracle_attention.argtypes = ([i32] * 9 + [dbl] + [P] * 7 + [i64, i64]
                                         + [P] + [P, i32, P, i32])
        lib.oracle_plan.restype = i32
        lib.oracle_plan.argtypes = [i32] * 9 + [P, P, P, i64, P, P, i64, P, P]
        lib.oracle_half_to_double.restype = dbl
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(int(bits))


def attention(w, subset=None, threads: int = 1, out: np.ndarray | None = None):
    """Attention of workload ``w`` in float64, shape [sum q, H, hv].

    ``subset``: iterable of sequence indices to compute (others stay 0).
    Returns ``(out, threads_used)``.
    """
    lib = _load()
    q = np.ascontiguousarray(w.query)
    kc = np.ascontiguousarray(w.key_cache)
    vc = np.ascontiguousarray(w.value_cache)
    bt = np.ascontiguousarray(w.block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(w.context_lens, dtype=np.int32)
    ql = np.ascontiguousarray(w.q_seqlens, dtype=np.int32)
    mask = None if w.mask is None else np.ascontiguousarray(w.mask)
    mask_q = mask_kv = 0
    if w.mask_type == 1:  # MASK_TYPE_NORM: [batch, max q, max_blocks_per_seq * block_size]
        assert mask.shape == (w.batch, w.max_seqlen_q, w.max_blocks_per_seq * w.block_size)
        mask_q, mask_kv = mask.shape[1], mask.shape[2]
    slopes = None if w.alibi_slopes is None else np.ascontiguousarray(w.alibi_slopes, dtype=np.float32)
    if out is None:
        out = np.zeros((w.total_q, w.num_heads, w.head_size_v), dtype=np.float64)
    sub = None if subset is None else np.ascontiguousarray(np.asarray(list(subset), dtype=np.int32))
    used = lib.oracle_attention(
        w.batch, w.num_heads, w.kv_heads, w.head_size_k, w.head_size_v, w.block_size,
        w.num_blocks, w.max_blocks_per_seq, w.mask_type, float(w.scale),
        _ptr(q.view(np.uint16)), _ptr(kc.view(np.uint16)), _ptr(vc.view(np.uint16)),
        _ptr(bt), _ptr(cl), _ptr(ql), None if mask is None else _ptr(mask.view(np.uint16)),
        mask_q, mask_kv, _ptr(slopes), _ptr(sub), 0 if sub is None else len(sub), _ptr(out), int(threads))
    if used < 0:
        raise ValueError("oracle: unsupported head size")
    return out, used


def plan(batch, num_heads, kv_heads, hk, hv, block_size, max_seqlen_q, chunk_blocks, num_sms,
         context_lens, q_seqlens=None):
    """The work list by the written rule: (work [n,8], combine [m,4], partial_rows)."""
    lib = _load()
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    ql = None if q_seqlens is None else np.ascontiguousarray(q_seqlens, dtype=np.int32)
    n_items, n_comb, prow = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    args = (batch, num_heads, kv_heads, hk, hv, block_size, max_seqlen_q, chunk_blocks, num_sms,
            _ptr(cl), _ptr(ql))
    lib.oracle_plan(*args, None, 0, ctypes.byref(n_items), None, 0, ctypes.byref(n_comb),
                    ctypes.byref(prow))
    work = np.zeros((n_items.value, 8), dtype=np.int32)
    comb = np.zeros((n_comb.value, 4), dtype=np.int32)
    rc = lib.oracle_plan(*args, _ptr(work), n_items.value, ctypes.byref(n_items), _ptr(comb),
                         n_comb.value, ctypes.byref(n_comb), ctypes.byref(prow))
    assert rc == 0
    return work, comb, int(prow.value)
