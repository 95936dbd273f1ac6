"""Python binding of libpa.so: GB300 PagedAttention forward.

The functions here marshal arguments to the C ABI declared in
``include/pa.h`` and raise :class:`PaError` on a non-OK status; every step of
the computation runs in the library's CUDA kernels. Device buffers are torch
tensors (torch supplies device memory and streams only). There is no CPU
fallback: if ``libpa.so`` has not been built, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from .build_lib import LIB

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_BUFFER_TOO_SMALL = 3
PA_ERR_CUDA = 4
PA_ERR_BLOCK_INDEX = 5
PA_ERR_TIMEOUT = 6

PA_MASK_NONE = 0
PA_MASK_NORM = 1
PA_MASK_ALIBI = 2
PA_MASK_SPEC = 4
PA_MASK_NORM_COMPRESS = 5

PA_WORK_INTS = 8
PA_COMBINE_INTS = 4
PA_STATUS_BYTES = 256
PA_FMA_MAX_ROWS = 8
PA_TC_TILE_ROWS = 64
PA_PF_TILE_ROWS = 128
PA_PF_PAIR_ROWS = 256

# Every symbol include/*.h declares (pa.h, the attention ABI; pa_probe.h, the
# HBM read probe; pa_testing.h, the test hook).
EXPORTS = ("pa_plan", "pa_forward", "pa_forward_noalloc", "pa_plan_bounds", "pa_plan_device",
           "pa_forward_device_plan", "pa_status_clear", "pa_status_read", "pa_status_string",
           "pa_hbm_read_probe", "pa_testing_set_wait_limit")
PA_PLAN_COUNTS = 4

PA_STATUS_BIT_BLOCK_INDEX = 1
PA_STATUS_BIT_TIMEOUT = 2
PA_STATUS_BIT_WORKSPACE = 4
PA_STATUS_BIT_PLAN = 8

# Size of the device array pa_forward_noalloc uses as its workspace.
PA_NOALLOC_SCRATCH_BYTES = 32 << 20


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class pa_config(ctypes.Structure):
    """Mirror of ``pa_config`` in include/pa.h."""

    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("head_size_k", ctypes.c_int32),
        ("head_size_v", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("max_seqlen_q", ctypes.c_int32),
        ("mask_type", ctypes.c_int32),
        ("chunk_blocks", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("scale", ctypes.c_float),
    ]


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libpa.so (built by ``build_lib.build``); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run paged_kv_cache_206_gb300.build_lib.build() "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    P, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(pa_config)
    lib.pa_plan.restype = ctypes.c_int
    lib.pa_plan.argtypes = [cfgp, P, P, P, i64, P, P, i64, P, P]
    lib.pa_forward.restype = ctypes.c_int
    lib.pa_forward.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, i64, P, i64, P, sz, P, P]
    lib.pa_forward_noalloc.restype = ctypes.c_int
    lib.pa_forward_noalloc.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, i64, P, i64, sz, P, P, P]
    lib.pa_plan_bounds.restype = ctypes.c_int
    lib.pa_plan_bounds.argtypes = [cfgp, P, P, P]
    lib.pa_plan_device.restype = ctypes.c_int
    lib.pa_plan_device.argtypes = [cfgp, P, P, P, i64, P, i64, P, P, P]
    lib.pa_forward_device_plan.restype = ctypes.c_int
    lib.pa_forward_device_plan.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, i64, P, i64, P, P, sz,
                                           P, P]
    lib.pa_status_clear.restype = ctypes.c_int
    lib.pa_status_clear.argtypes = [P, P]
    lib.pa_status_read.restype = ctypes.c_int
    lib.pa_status_read.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_hbm_read_probe.restype = ctypes.c_int
    lib.pa_hbm_read_probe.argtypes = [P, sz, ctypes.c_int, P, P]
    lib.pa_testing_set_wait_limit.restype = ctypes.c_int
    lib.pa_testing_set_wait_limit.argtypes = [ctypes.c_longlong]
    if path == LIB:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().pa_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != PA_OK:
        raise PaError(status, where)


def make_config(*, batch, num_heads, kv_heads, head_size_k, head_size_v=None, block_size,
                num_blocks, max_blocks_per_seq, max_seqlen_q=1, mask_type=PA_MASK_NONE,
                chunk_blocks=0, num_sms=0, scale=0.0) -> pa_config:
    return pa_config(int(batch), int(num_heads), int(kv_heads), int(head_size_k),
                     int(head_size_k if head_size_v is None else head_size_v), int(block_size),
                     int(num_blocks), int(max_blocks_per_seq), int(max_seqlen_q),
                     int(mask_type), int(chunk_blocks), int(num_sms), float(scale))


def config_for(w, num_sms: int = 0, chunk_blocks: int | None = None) -> pa_config:
    """pa_config of a ``workloads.Workload``."""
    return make_config(batch=w.batch, num_heads=w.num_heads, kv_heads=w.kv_heads,
                       head_size_k=w.head_size_k, head_size_v=w.head_size_v,
                       block_size=w.block_size, num_blocks=w.num_blocks,
                       max_blocks_per_seq=w.max_blocks_per_seq, max_seqlen_q=w.max_seqlen_q,
                       mask_type=w.mask_type,
                       chunk_blocks=w.chunk_blocks if chunk_blocks is None else chunk_blocks,
                       num_sms=num_sms, scale=w.scale)


@dataclass
class Plan:
    work: np.ndarray  # int32 [n_items, 8]
    combine: np.ndarray  # int32 [n_combine, 4]
    workspace_bytes: int


def _np_ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def pa_plan(cfg: pa_config, context_lens, q_seqlens=None) -> Plan:
    """Host planner (pa_plan): validate and build the work and combine lists."""
    lib = load_library()
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    ql = None if q_seqlens is None else np.ascontiguousarray(q_seqlens, dtype=np.int32)
    n_items, n_comb, ws = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
    _check(lib.pa_plan(ctypes.byref(cfg), _np_ptr(cl), _np_ptr(ql), None, 0, ctypes.byref(n_items),
                       None, 0, ctypes.byref(n_comb), ctypes.byref(ws)), "pa_plan")
    work = np.zeros((n_items.value, PA_WORK_INTS), dtype=np.int32)
    comb = np.zeros((max(n_comb.value, 0), PA_COMBINE_INTS), dtype=np.int32)
    _check(lib.pa_plan(ctypes.byref(cfg), _np_ptr(cl), _np_ptr(ql), _np_ptr(work), n_items.value,
                       ctypes.byref(n_items), _np_ptr(comb), n_comb.value, ctypes.byref(n_comb),
                       ctypes.byref(ws)), "pa_plan")
    return Plan(work, comb, int(ws.value))


def _tptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def pa_forward(cfg: pa_config, query, key_cache, value_cache, block_tables, context_lens,
               q_seqlens, mask, alibi_slopes, work, combine, workspace, out, stream=None) -> None:
    """Enqueue attention (pa_forward). All tensor arguments are CUDA tensors
    (``q_seqlens``, ``mask``, ``alibi_slopes`` and ``combine`` may be None)."""
    lib = load_library()
    n_items = 0 if work is None else work.shape[0]
    n_comb = 0 if combine is None else combine.shape[0]
    st = lib.pa_forward(ctypes.byref(cfg), _tptr(query), _tptr(key_cache), _tptr(value_cache),
                        _tptr(block_tables), _tptr(context_lens), _tptr(q_seqlens), _tptr(mask),
                        _tptr(alibi_slopes), _tptr(work), n_items,
                        _tptr(combine) if n_comb else None, n_comb, _tptr(workspace),
                        workspace.numel() * workspace.element_size(), _tptr(out),
                        _stream_handle(stream))
    _check(st, "pa_forward")


def pa_forward_noalloc(cfg: pa_config, query, key_cache, value_cache, block_tables,
                       context_lens, q_seqlens, mask, alibi_slopes, work, combine,
                       workspace_bytes: int, status, out, stream=None) -> None:
    """Enqueue attention without a workspace argument (pa_forward_noalloc): for
    callers that cannot allocate device memory, the library's own fixed device
    array serves as the workspace. ``workspace_bytes`` is what pa_plan
    reported; ``status`` is a CUDA uint32/int32 tensor of one element, or None."""
    lib = load_library()
    n_items = 0 if work is None else work.shape[0]
    n_comb = 0 if combine is None else combine.shape[0]
    st = lib.pa_forward_noalloc(ctypes.byref(cfg), _tptr(query), _tptr(key_cache),
                                _tptr(value_cache), _tptr(block_tables), _tptr(context_lens),
                                _tptr(q_seqlens), _tptr(mask), _tptr(alibi_slopes), _tptr(work),
                                n_items, _tptr(combine) if n_comb else None, n_comb,
                                int(workspace_bytes), _tptr(status), _tptr(out),
                                _stream_handle(stream))
    _check(st, "pa_forward_noalloc")


def hbm_read_probe(buf, ctas_per_sm: int, sink, stream=None) -> None:
    """Enqueue one streaming read of the CUDA tensor ``buf`` (pa_hbm_read_probe);
    ``sink`` is a one-element CUDA int32/uint32 tensor the probe XORs into."""
    _check(load_library().pa_hbm_read_probe(_tptr(buf), buf.numel() * buf.element_size(),
                                            int(ctas_per_sm), _tptr(sink),
                                            _stream_handle(stream)), "pa_hbm_read_probe")


def testing_set_wait_limit(cycles: int) -> None:
    """Test hook (pa_testing_set_wait_limit): the cycle limit of the decode
    kernels' waits on other roles for later launches; 0 restores the default."""
    _check(load_library().pa_testing_set_wait_limit(int(cycles)), "pa_testing_set_wait_limit")


def pa_status_clear(workspace, stream=None) -> None:
    _check(load_library().pa_status_clear(_tptr(workspace), _stream_handle(stream)),
           "pa_status_clear")


def pa_status_read(workspace, stream=None) -> tuple[int, int]:
    """(status, bits): waits for the stream and reads the kernels' status word."""
    bits = ctypes.c_uint32()
    st = load_library().pa_status_read(_tptr(workspace), _stream_handle(stream), ctypes.byref(bits))
    return st, bits.value


class DeviceBatch:
    """A workload's tensors on one CUDA device, planned and ready to run.

    Holds the device copies of the inputs, the work and combine lists, the
    workspace (status word cleared) and the output buffer.
    """

    def __init__(self, w, device="cuda", num_sms: int | None = None,
                 chunk_blocks: int | None = None):
        import torch
        dev = torch.device(device)
        if num_sms is None:
            num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
        self.w = w
        self.cfg = config_for(w, num_sms=num_sms, chunk_blocks=chunk_blocks)
        ql_host = None if np.all(w.q_seqlens == 1) else w.q_seqlens
        self.plan = pa_plan(self.cfg, w.context_lens, ql_host)

        def up(a, dtype=None):
            if a is None:
                return None
            t = torch.from_numpy(np.ascontiguousarray(a))
            return t.to(dev, non_blocking=False)

        self.query = up(w.query)
        self.key_cache = up(w.key_cache)
        # shared-KV cache: the value pointer is the key cache itself
        self.value_cache = self.key_cache if w.shared_kv else up(w.value_cache)
        self.block_tables = up(w.block_tables)
        self.context_lens = up(w.context_lens)
        self.q_seqlens = up(ql_host)
        self.mask = up(w.mask)
        self.alibi_slopes = up(w.alibi_slopes)
        self.work = up(self.plan.work)
        self.combine = up(self.plan.combine) if self.plan.combine.shape[0] else None
        ws = max(self.plan.workspace_bytes, PA_STATUS_BYTES)
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)
        self.out = torch.empty((w.total_q, w.num_heads, w.head_size_v), dtype=torch.float16,
                               device=dev)

    def forward(self, stream=None):
        pa_forward(self.cfg, self.query, self.key_cache, self.value_cache, self.block_tables,
                   self.context_lens, self.q_seqlens, self.mask, self.alibi_slopes, self.work,
                   self.combine, self.workspace, self.out, stream)
        return self.out

    def status(self, stream=None):
        return pa_status_read(self.workspace, stream)


def _align(n: int, a: int = 256) -> int:
    return (n + a - 1) // a * a


def list_capacity(cfg: pa_config) -> tuple[int, int]:
    """(work items, combine entries) that hold pa_plan's lists for any context
    and query lengths the configuration admits.

    A (sequence, kv head) has at most QT = ceil(G * max_seqlen_q / TR) query
    tiles, so there are at most B * Hk * QT combine entries. With an explicit
    chunk c each tile has at most ceil(max_blocks_per_seq / c) splits; with the
    automatic rule c >= W / (8 * num_sms), so the items, a sum over tiles of
    ceil(NB / c) <= NB / c + 1, number at most 8 * num_sms + B * Hk * QT.
    """
    rows = (cfg.num_heads // cfg.kv_heads) * max(1, cfg.max_seqlen_q)
    pf_heads = cfg.head_size_k == cfg.head_size_v and cfg.head_size_k in (64, 128)
    if rows <= PA_FMA_MAX_ROWS:
        tr = rows
    elif rows > PA_TC_TILE_ROWS and pf_heads:
        tr = PA_PF_PAIR_ROWS if rows > PA_PF_TILE_ROWS else PA_PF_TILE_ROWS
    else:
        tr = PA_TC_TILE_ROWS
    tiles = cfg.batch * cfg.kv_heads * (-(-rows // tr))
    if cfg.chunk_blocks > 0:
        items = tiles * (-(-cfg.max_blocks_per_seq // cfg.chunk_blocks))
    else:
        items = 8 * cfg.num_sms + tiles
    return items, tiles


# Outputs up to this size are stored by the kernels straight into pinned host
# memory (no copy node: about 10 us less per step for a decode batch); larger
# ones go to a device buffer and one copy, since the kernels' scattered stores
# over the host link are slower than the copy engine at volume (a 67 MB
# prefill output took 1.7 ms that way, against 0.35 ms for the copy).
ZERO_COPY_OUT_BYTES = 4 << 20


def _device_out(out, dev):
    """A device buffer for ``out``, or None when the kernels write it directly."""
    import torch
    if out.numel() * out.element_size() <= ZERO_COPY_OUT_BYTES:
        return None
    return torch.empty(out.shape, dtype=out.dtype, device=dev)


class HostStep:
    """One attention step whose per-step inputs live in pinned host memory.

    The caller writes the step's query, block tables, context lengths (and
    query lengths) into the pinned views ``query``, ``block_tables``,
    ``context_lens`` and ``q_seqlens``; :meth:`run` then plans the step
    (pa_plan, writing the work and combine lists straight into the same pinned
    arena), moves the used part of the arena to the device with one
    host-to-device copy, enqueues pa_forward on device pointers into it and
    waits for the stream. An output of at most ``ZERO_COPY_OUT_BYTES`` is
    stored by the kernels straight into the pinned ``out`` tensor; a larger
    one goes to a device buffer and is copied back. The KV cache, mask and
    ALiBi slopes stay resident on the device.
    """

    def __init__(self, cfg: pa_config, key_cache, value_cache, total_q: int, mask=None,
                 alibi_slopes=None, device=None):
        import torch
        self.cfg = cfg
        dev = key_cache.device if device is None else torch.device(device)
        self.key_cache, self.value_cache = key_cache, value_cache
        self.mask, self.alibi_slopes = mask, alibi_slopes
        B, H, hk, hv = cfg.batch, cfg.num_heads, cfg.head_size_k, cfg.head_size_v
        has_ql = cfg.max_seqlen_q > 1
        self.total_q = int(total_q)
        self.work_cap, ccap = list_capacity(cfg)
        self.combine_cap = max(ccap, 1)
        # The combine list sits before the work list so that the copied
        # prefix ends with the items actually planned.
        sizes = [("query", self.total_q * H * hk * 2),
                 ("block_tables", B * cfg.max_blocks_per_seq * 4),
                 ("context_lens", B * 4), ("q_seqlens", B * 4 if has_ql else 0),
                 ("combine", self.combine_cap * PA_COMBINE_INTS * 4),
                 ("work", self.work_cap * PA_WORK_INTS * 4)]
        self.offsets, off = {}, 0
        for name, n in sizes:
            self.offsets[name] = off
            off = _align(off + n)
        self.arena_bytes = off
        self.h_arena = torch.zeros(off, dtype=torch.uint8).pin_memory()
        self.d_arena = torch.zeros(off, dtype=torch.uint8, device=dev)

        def hview(name, dtype, shape):
            o = self.offsets[name]
            n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            return self.h_arena[o:o + n].view(dtype).view(shape)

        self.query = hview("query", torch.float16, (self.total_q, H, hk))
        self.block_tables = hview("block_tables", torch.int32, (B, cfg.max_blocks_per_seq))
        self.context_lens = hview("context_lens", torch.int32, (B,))
        self.q_seqlens = hview("q_seqlens", torch.int32, (B,)) if has_ql else None
        self.out = torch.empty((self.total_q, H, hv), dtype=torch.float16).pin_memory()
        self.d_out = _device_out(self.out, dev)
        self._d = {k: self.d_arena.data_ptr() + v for k, v in self.offsets.items()}
        self._h = {k: self.h_arena.data_ptr() + v for k, v in self.offsets.items()}
        self.workspace = None
        self.last_h2d_bytes = 0
        self.n_items = self.n_combine = 0

    def run(self, stream=None):
        """Plan, copy in, attend (into the pinned ``out`` tensor, or a device
        buffer copied into it); returns ``out``."""
        import torch
        lib = load_library()
        cfg, h, d, P = self.cfg, self._h, self._d, ctypes.c_void_p
        has_ql = self.q_seqlens is not None
        n_items, n_comb, ws = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
        _check(lib.pa_plan(ctypes.byref(cfg), P(h["context_lens"]),
                           P(h["q_seqlens"]) if has_ql else None, P(h["work"]), self.work_cap,
                           ctypes.byref(n_items), P(h["combine"]), self.combine_cap,
                           ctypes.byref(n_comb), ctypes.byref(ws)), "pa_plan")
        self.n_items, self.n_combine = n_items.value, n_comb.value
        need = max(int(ws.value), PA_STATUS_BYTES)
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = torch.zeros(need, dtype=torch.uint8, device=self.d_arena.device)
        used = self.offsets["work"] + self.n_items * PA_WORK_INTS * 4
        self.last_h2d_bytes = used
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            self.d_arena[:used].copy_(self.h_arena[:used], non_blocking=True)
        st = lib.pa_forward(ctypes.byref(cfg), P(d["query"]), _tptr(self.key_cache),
                            _tptr(self.value_cache), P(d["block_tables"]), P(d["context_lens"]),
                            P(d["q_seqlens"]) if has_ql else None, _tptr(self.mask),
                            _tptr(self.alibi_slopes), P(d["work"]), self.n_items,
                            P(d["combine"]) if self.n_combine else None, self.n_combine,
                            _tptr(self.workspace), self.workspace.numel(),
                            _tptr(self.out if self.d_out is None else self.d_out),
                            ctypes.c_void_p(s.cuda_stream))
        _check(st, "pa_forward")
        if self.d_out is not None:
            with torch.cuda.stream(s):
                self.out.copy_(self.d_out, non_blocking=True)
        s.synchronize()
        return self.out

    def status(self, stream=None):
        return pa_status_read(self.workspace, stream)


def pa_plan_bounds(cfg: pa_config) -> tuple[int, int, int]:
    """(work_cap, comb_cap, workspace_bytes) that hold any plan of ``cfg``."""
    w, c, ws = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
    _check(load_library().pa_plan_bounds(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(c),
                                         ctypes.byref(ws)), "pa_plan_bounds")
    return w.value, c.value, ws.value


class DevicePlanStep:
    """A decode step planned on the device: pa_plan_device, then
    pa_forward_device_plan, both on device tensors, with list buffers sized by
    pa_plan_bounds. The launches do not depend on the lengths, so ``run`` may
    be recorded in a CUDA graph and replayed after ``context_lens`` (and
    ``q_seqlens``) are updated in place."""

    def __init__(self, db: "DeviceBatch"):
        import torch
        self.db = db
        dev = db.key_cache.device
        self.work_cap, self.comb_cap, ws = pa_plan_bounds(db.cfg)
        self.work = torch.zeros((self.work_cap, PA_WORK_INTS), dtype=torch.int32, device=dev)
        self.combine = torch.zeros((max(self.comb_cap, 1), PA_COMBINE_INTS), dtype=torch.int32,
                                   device=dev)
        self.counts = torch.zeros(PA_PLAN_COUNTS, dtype=torch.int32, device=dev)
        self.workspace = torch.zeros(max(ws, PA_STATUS_BYTES), dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(db.out)

    def plan(self, stream=None):
        db = self.db
        _check(load_library().pa_plan_device(
            ctypes.byref(db.cfg), _tptr(db.context_lens), _tptr(db.q_seqlens), _tptr(self.work),
            self.work_cap, _tptr(self.combine), self.comb_cap, _tptr(self.counts),
            _tptr(self.workspace), _stream_handle(stream)), "pa_plan_device")

    def forward(self, stream=None):
        db = self.db
        _check(load_library().pa_forward_device_plan(
            ctypes.byref(db.cfg), _tptr(db.query), _tptr(db.key_cache), _tptr(db.value_cache),
            _tptr(db.block_tables), _tptr(db.context_lens), _tptr(db.q_seqlens), _tptr(db.mask),
            _tptr(db.alibi_slopes), _tptr(self.work), self.work_cap, _tptr(self.combine),
            self.comb_cap, _tptr(self.counts), _tptr(self.workspace), self.workspace.numel(),
            _tptr(self.out), _stream_handle(stream)), "pa_forward_device_plan")

    def run(self, stream=None):
        self.plan(stream)
        self.forward(stream)
        return self.out

    def status(self, stream=None):
        return pa_status_read(self.workspace, stream)


class GraphStep:
    """One attention step recorded once as a CUDA graph and replayed per step.

    The step's inputs live in one pinned host arena (views ``context_lens``,
    ``q_seqlens``, ``query``, ``block_tables``). The graph holds: the device
    planner (pa_plan_device), reading the lengths straight from the pinned
    arena (mapped into the device's address space), beside it on a second
    stream the host-to-device copy of the arena, then the forward pass over
    the planner's lists (pa_forward_device_plan), whose output is the pinned
    ``out`` tensor itself when it is at most ``ZERO_COPY_OUT_BYTES`` (the
    kernels store the result straight into host memory), else a device buffer
    copied into ``out``. :meth:`run` replays it and waits, so a decode loop
    costs one graph launch per step.
    The launches do not depend on the lengths (grids are pa_plan_bounds'
    capacities), which is what allows the recording.
    """

    def __init__(self, cfg: pa_config, key_cache, value_cache, total_q: int, mask=None,
                 alibi_slopes=None):
        import torch
        self.cfg = cfg
        dev = key_cache.device
        self.key_cache, self.value_cache = key_cache, value_cache
        self.mask, self.alibi_slopes = mask, alibi_slopes
        B, H, hk, hv = cfg.batch, cfg.num_heads, cfg.head_size_k, cfg.head_size_v
        has_ql = cfg.max_seqlen_q > 1
        self.total_q = int(total_q)
        sizes = [("context_lens", B * 4), ("q_seqlens", B * 4 if has_ql else 0),
                 ("query", self.total_q * H * hk * 2),
                 ("block_tables", B * cfg.max_blocks_per_seq * 4)]
        self.offsets, off = {}, 0
        for name, n in sizes:
            self.offsets[name] = off
            off = _align(off + n)
        self.arena_bytes = off
        self.h_arena = torch.zeros(off, dtype=torch.uint8).pin_memory()
        self.d_arena = torch.zeros(off, dtype=torch.uint8, device=dev)

        def view(t, name, dtype, shape):
            o = self.offsets[name]
            n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            return t[o:o + n].view(dtype).view(shape)

        self.query = view(self.h_arena, "query", torch.float16, (self.total_q, H, hk))
        self.block_tables = view(self.h_arena, "block_tables", torch.int32, (B, cfg.max_blocks_per_seq))
        self.context_lens = view(self.h_arena, "context_lens", torch.int32, (B,))
        self.q_seqlens = view(self.h_arena, "q_seqlens", torch.int32, (B,)) if has_ql else None
        self._dq = view(self.d_arena, "query", torch.float16, (self.total_q, H, hk))
        self._dbt = view(self.d_arena, "block_tables", torch.int32, (B, cfg.max_blocks_per_seq))
        self._dcl = view(self.d_arena, "context_lens", torch.int32, (B,))
        self._dql = view(self.d_arena, "q_seqlens", torch.int32, (B,)) if has_ql else None
        self.work_cap, self.comb_cap, ws = pa_plan_bounds(cfg)
        self.work = torch.zeros((self.work_cap, PA_WORK_INTS), dtype=torch.int32, device=dev)
        self.combine = torch.zeros((max(self.comb_cap, 1), PA_COMBINE_INTS), dtype=torch.int32,
                                   device=dev)
        self.counts = torch.zeros(PA_PLAN_COUNTS, dtype=torch.int32, device=dev)
        self.workspace = torch.zeros(max(ws, PA_STATUS_BYTES), dtype=torch.uint8, device=dev)
        self.out = torch.empty((self.total_q, H, hv), dtype=torch.float16).pin_memory()
        self.d_out = _device_out(self.out, dev)
        self.h2d_bytes = self.arena_bytes
        self.stream = torch.cuda.Stream(device=dev)
        self.side_stream = torch.cuda.Stream(device=dev)
        self.graph = None

    def _enqueue(self, events=None):
        """Enqueue the step on its stream. Without ``events`` (the recorded
        graph), the copy of the query and block tables runs on a second stream
        beside the device planner, which needs only the lengths. With
        ``events`` (five CUDA events) the stages run one after another, an event
        recorded before the host-to-device copy and after each stage (copy in,
        device planner, attention and combine, copy out: empty when the kernels
        write the pinned output themselves), to time them separately."""
        import torch
        lib, cfg, s = load_library(), self.cfg, self.stream

        def mark(k):
            if events is not None:
                events[k].record(s)

        def plan(cl, ql):
            _check(lib.pa_plan_device(
                ctypes.byref(cfg), _tptr(cl), _tptr(ql), _tptr(self.work),
                self.work_cap, _tptr(self.combine), self.comb_cap, _tptr(self.counts),
                _tptr(self.workspace), ctypes.c_void_p(s.cuda_stream)), "pa_plan_device")

        mark(0)
        if events is None:
            # the planner reads the lengths from the pinned arena itself (a
            # few KB over the host link) while the arena's copy, which the
            # forward pass needs, runs beside it
            side = self.side_stream
            side.wait_stream(s)
            plan(self.context_lens, self.q_seqlens)
            with torch.cuda.stream(side):
                self.d_arena.copy_(self.h_arena, non_blocking=True)
            s.wait_stream(side)
        else:
            with torch.cuda.stream(s):
                self.d_arena.copy_(self.h_arena, non_blocking=True)
            mark(1)
            plan(self._dcl, self._dql)
        mark(2)
        _check(lib.pa_forward_device_plan(
            ctypes.byref(cfg), _tptr(self._dq), _tptr(self.key_cache), _tptr(self.value_cache),
            _tptr(self._dbt), _tptr(self._dcl), _tptr(self._dql), _tptr(self.mask),
            _tptr(self.alibi_slopes), _tptr(self.work), self.work_cap, _tptr(self.combine),
            self.comb_cap, _tptr(self.counts), _tptr(self.workspace), self.workspace.numel(),
            _tptr(self.out if self.d_out is None else self.d_out),
            ctypes.c_void_p(s.cuda_stream)), "pa_forward_device_plan")
        mark(3)
        if self.d_out is not None:
            with torch.cuda.stream(s):
                self.out.copy_(self.d_out, non_blocking=True)
        mark(4)

    def record(self):
        """Run the step once directly (kernel attributes and tensor maps are set
        up then), then record it as a graph."""
        import torch
        self._enqueue()
        self.stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self._enqueue()
        self.graph = g

    def run_stages(self, events):
        """Run the step's stages directly (no graph), recording ``events`` (five
        CUDA events) around them for timing each stage, and wait."""
        self._enqueue(events)
        self.stream.synchronize()
        return self.out

    def run(self):
        """Replay the step and wait for it; returns the pinned ``out`` tensor."""
        import torch
        if self.graph is None:
            self.record()
        # replay() launches on the current stream: make that the step's own
        with torch.cuda.stream(self.stream):
            self.graph.replay()
        self.stream.synchronize()
        return self.out

    def status(self):
        return pa_status_read(self.workspace, self.stream)
