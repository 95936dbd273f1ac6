"""The C ABI of libpa.so on a machine without a GPU: the library loads, exports
every function that include/*.h declares, and rejects bad arguments on the host
before it touches CUDA."""
import ctypes
import glob
import os
import re
import subprocess

import numpy as np
import pytest

import paged_kv_cache_206_gb300 as pa
from paged_kv_cache_206_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return pa.load_library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        names |= set(re.findall(r"\b(pa_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(pa.EXPORTS) <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", build_lib.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_library_does_not_link_the_driver(lib):
    out = subprocess.run(["ldd", build_lib.LIB], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_status_strings(lib):
    for s in range(7):
        assert pa.status_string(s) not in ("", "unknown status")
    assert pa.status_string(99) == "unknown status"


def _cfg(**kw):
    base = dict(batch=1, num_heads=4, kv_heads=4, head_size_k=64, block_size=16, num_blocks=4,
                max_blocks_per_seq=4, num_sms=1)
    base.update(kw)
    return pa.make_config(**base)


def _fwd(lib, cfg, **ptrs):
    """Call pa_forward with fake, aligned non-null addresses unless overridden."""
    fake = ctypes.c_void_p(1 << 20)
    args = dict(query=fake, key=fake, value=fake, bt=fake, ctx=fake, ql=None, mask=None,
                slopes=None, work=fake, n_items=1, comb=None, n_comb=0, ws=fake, ws_bytes=256,
                out=fake)
    args.update(ptrs)
    return lib.pa_forward(ctypes.byref(cfg), args["query"], args["key"], args["value"], args["bt"],
                          args["ctx"], args["ql"], args["mask"], args["slopes"], args["work"],
                          args["n_items"], args["comb"], args["n_comb"], args["ws"],
                          args["ws_bytes"], args["out"], None)


def test_forward_host_checks(lib):
    c = _cfg()
    fake = ctypes.c_void_p(1 << 20)
    assert _fwd(lib, c, query=None) == pa.PA_ERR_INVALID_ARG
    assert _fwd(lib, c, ws=None) == pa.PA_ERR_INVALID_ARG
    assert _fwd(lib, c, mask=fake) == pa.PA_ERR_INVALID_ARG          # mask only with NORM_COMPRESS
    assert _fwd(lib, _cfg(mask_type=5)) == pa.PA_ERR_INVALID_ARG     # NORM_COMPRESS needs a mask
    assert _fwd(lib, _cfg(mask_type=2)) == pa.PA_ERR_INVALID_ARG     # ALIBI needs slopes
    assert _fwd(lib, _cfg(mask_type=1)) == pa.PA_ERR_INVALID_ARG     # NORM needs its mask
    assert _fwd(lib, _cfg(mask_type=1), mask=fake, n_items=0, work=None) == pa.PA_OK
    assert _fwd(lib, c, slopes=fake) == pa.PA_ERR_INVALID_ARG
    assert _fwd(lib, _cfg(mask_type=4)) == pa.PA_ERR_UNSUPPORTED
    assert _fwd(lib, _cfg(block_size=8)) == pa.PA_ERR_INVALID_ARG
    assert _fwd(lib, c, key=ctypes.c_void_p((1 << 20) + 8)) == pa.PA_ERR_INVALID_ARG  # 16-B align
    assert _fwd(lib, c, ws=ctypes.c_void_p((1 << 20) + 16)) == pa.PA_ERR_INVALID_ARG  # 256-B align
    assert _fwd(lib, c, ws_bytes=255) == pa.PA_ERR_BUFFER_TOO_SMALL
    assert _fwd(lib, c, n_comb=1, comb=None) == pa.PA_ERR_INVALID_ARG
    assert _fwd(lib, c, n_items=-1) == pa.PA_ERR_INVALID_ARG
    assert _fwd(lib, c, n_items=0, work=None) == pa.PA_OK              # nothing to do
    # value_cache == key_cache is the shared-KV layout: V = first hv dims of a
    # K row, so hv may not exceed hk; distinct caches have no such rule
    wide_v = _cfg(head_size_v=128)
    assert _fwd(lib, wide_v, n_items=0, work=None) == pa.PA_ERR_INVALID_ARG
    other = ctypes.c_void_p((1 << 21))
    assert _fwd(lib, wide_v, value=other, n_items=0, work=None) == pa.PA_OK
    assert lib.pa_status_clear(None, None) == pa.PA_ERR_INVALID_ARG


def test_plan_bounds_and_device_plan_host_checks(lib):
    import numpy as np
    for kw in (dict(), dict(max_seqlen_q=3, num_heads=16, kv_heads=1), dict(chunk_blocks=3),
               dict(batch=7, max_blocks_per_seq=40, num_sms=152)):
        c = _cfg(**kw)
        w, m, ws = pa.pa_plan_bounds(c)
        assert (w, m) == pa.list_capacity(c)
        rows = (c.num_heads // c.kv_heads) * max(1, c.max_seqlen_q)
        tr = rows if rows <= 8 else 64
        up = lambda x: (x + 255) // 256 * 256
        assert ws == up(up(256 + w * tr * c.head_size_v * 2) + w * tr * 4)
    fake = ctypes.c_void_p(1 << 20)
    c = _cfg()

    def dev(cfg, **kw):
        a = dict(ctx=fake, ql=None, work=fake, wcap=4, comb=fake, ccap=4, counts=fake, ws=fake)
        a.update(kw)
        return lib.pa_plan_device(ctypes.byref(cfg), a["ctx"], a["ql"], a["work"], a["wcap"],
                                  a["comb"], a["ccap"], a["counts"], a["ws"], None)
    assert dev(c, ctx=None) == pa.PA_ERR_INVALID_ARG
    assert dev(c, counts=None) == pa.PA_ERR_INVALID_ARG
    assert dev(c, wcap=0) == pa.PA_ERR_INVALID_ARG
    assert dev(c, comb=None) == pa.PA_ERR_INVALID_ARG
    assert dev(c, ws=ctypes.c_void_p((1 << 20) + 64)) == pa.PA_ERR_INVALID_ARG
    assert dev(c, work=ctypes.c_void_p((1 << 20) + 4)) == pa.PA_ERR_INVALID_ARG  # 16-byte stores
    assert dev(c, comb=ctypes.c_void_p((1 << 20) + 8)) == pa.PA_ERR_INVALID_ARG
    assert dev(_cfg(block_size=8)) == pa.PA_ERR_INVALID_ARG
    assert dev(_cfg(mask_type=4)) == pa.PA_ERR_UNSUPPORTED
    # the automatic chunk rule needs the SM count (the device planner divides by it)
    assert dev(_cfg(chunk_blocks=0, num_sms=0)) == pa.PA_ERR_INVALID_ARG
    assert dev(_cfg(chunk_blocks=-1)) == pa.PA_ERR_INVALID_ARG
    w_, c_, s_ = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
    for bad in (_cfg(chunk_blocks=0, num_sms=0), _cfg(chunk_blocks=-1)):
        assert lib.pa_plan_bounds(ctypes.byref(bad), ctypes.byref(w_), ctypes.byref(c_),
                                  ctypes.byref(s_)) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_forward_device_plan(ctypes.byref(c), fake, fake, fake, fake, fake, None, None,
                                      None, fake, 4, None, 0, None, fake, 256, fake,
                                      None) == pa.PA_ERR_INVALID_ARG  # counts required
    assert lib.pa_status_read(None, None, None) == pa.PA_ERR_INVALID_ARG


def _header_define(name):
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    m = re.search(r"^#define\s+" + name + r"\s+(.+)$", text, re.M)
    assert m, name
    expr = re.sub(r"/\*.*?\*/", "", m.group(1)).strip()
    expr = re.sub(r"(\d+)u\b", r"\1", expr)  # C unsigned suffixes
    assert re.fullmatch(r"[0-9()<< +*x]+", expr), expr
    return int(eval(expr))


def test_binding_constants_match_the_header():
    """The binding restates some of pa.h's #defines; they must agree."""
    for name in ("PA_NOALLOC_SCRATCH_BYTES", "PA_STATUS_BYTES", "PA_WORK_INTS",
                 "PA_COMBINE_INTS", "PA_FMA_MAX_ROWS", "PA_TC_TILE_ROWS", "PA_PF_TILE_ROWS",
                 "PA_PF_PAIR_ROWS", "PA_PLAN_COUNTS", "PA_STATUS_BIT_BLOCK_INDEX",
                 "PA_STATUS_BIT_TIMEOUT", "PA_STATUS_BIT_WORKSPACE", "PA_STATUS_BIT_PLAN"):
        assert getattr(pa, name) == _header_define(name), name


def test_probe_and_testing_hook_host_checks(lib):
    fake = ctypes.c_void_p(1 << 20)
    probe = lib.pa_hbm_read_probe
    assert probe(None, 1024, 1, fake, None) == pa.PA_ERR_INVALID_ARG
    assert probe(fake, 0, 1, fake, None) == pa.PA_ERR_INVALID_ARG
    assert probe(fake, 1000, 1, fake, None) == pa.PA_ERR_INVALID_ARG       # not a multiple of 32
    assert probe(ctypes.c_void_p((1 << 20) + 16), 1024, 1, fake, None) == pa.PA_ERR_INVALID_ARG
    assert probe(fake, 1024, 0, fake, None) == pa.PA_ERR_INVALID_ARG
    assert probe(fake, 1024, 9, fake, None) == pa.PA_ERR_INVALID_ARG
    assert probe(fake, 1024, 1, None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_testing_set_wait_limit(-1) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_testing_set_wait_limit(0) == pa.PA_OK


def test_noalloc_rejects_bad_arguments_before_enqueueing(lib):
    """pa_forward_noalloc runs pa_forward's host checks before it touches the
    stream: with no CUDA device, a call that passed them would fail in the
    CUDA runtime instead (PA_ERR_CUDA), so every bad call here must come back
    PA_ERR_INVALID_ARG."""
    c = _cfg()
    fake = ctypes.c_void_p(1 << 20)

    def call(**kw):
        a = dict(query=fake, key=fake, value=fake, bt=fake, ctx=fake, mask=None, slopes=None,
                 work=fake, n_items=1, ws_bytes=256, out=fake)
        a.update(kw)
        return lib.pa_forward_noalloc(ctypes.byref(c), a["query"], a["key"], a["value"], a["bt"],
                                      a["ctx"], None, a["mask"], a["slopes"], a["work"],
                                      a["n_items"], None, 0, a["ws_bytes"], None, a["out"], None)
    assert call(query=None) == pa.PA_ERR_INVALID_ARG
    assert call(out=ctypes.c_void_p((1 << 20) + 2)) == pa.PA_ERR_INVALID_ARG
    assert call(mask=fake) == pa.PA_ERR_INVALID_ARG
    assert call(work=None) == pa.PA_ERR_INVALID_ARG
    assert call(ws_bytes=pa.PA_NOALLOC_SCRATCH_BYTES + 1) == pa.PA_ERR_BUFFER_TOO_SMALL
