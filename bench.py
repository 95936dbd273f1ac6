"""Benchmark: paged-attention effective KV HBM GB/s and query tokens/s.

One step is one pass of the whole device path over one synthetic batch:
pa_forward over the planned work list (the attention kernel, then the split-KV
combine kernel when the plan has split tiles). The work list comes from
pa_plan before the timed region (host code, timed separately as plan_us).
The end-to-end number (`e2e`) starts from pinned host buffers: each timed
step replays one recorded CUDA graph that copies the step's inputs to the
device, plans on the device and runs attention, whose kernels store an
output of up to 4 MiB straight into a pinned host tensor (a larger one is
copied back from device memory; device-to-host bytes are the output's size
either way), and the host waits for it. The same step planned
on the host with direct launches is reported beside it (`e2e.host_planned`),
and the graph's stages are timed one by one with CUDA events
(`e2e.breakdown_us`).

One run measures every workload of the benchmark table (`configs`): tiny,
GQA, parallel/speculative and ALiBi decode, long-context MQA split-KV, plus
MLA-style shared-KV decode and causal prefill. The headline line is ALiBi
decode (B=128, H=Hk=40, hk=hv=128, block_size=128, lengths uniform in
[1, 2048], ALiBi slopes), the largest single-GPU workload (2.62 GB of KV);
`--workload NAME` measures that one alone. Before every timed step the
129 MB L2 is flushed outside the timed events (a 512 MB buffer is written,
then half of it read back so the write-backs of the flush's dirty lines also
happen before the events), so every step reads the KV cache from HBM.

The HBM read ceiling is measured in the same process: a streaming read of
2 GiB (pa_hbm_read_probe), best of several grid shapes. Roofline fractions are
given against it (`frac_read`) and against the measured copy
(`frac`, MEASURED_PEAKS.json).

`--impl reference` times the CPU oracle on this machine's cores instead, on a
bounded sample of the headline workload, and prints the same JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn effective KV HBM GB/s (% of GB300 peak) and query tokens/s"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TFLOPS = 1900.0
FLUSH_BYTES = 512 << 20
REF_BUDGET_S = 150.0  # the reference arm's whole run, about
READ_PROBE_BYTES = 2 << 30

# Every workload of the benchmark table, in the order of the table; the rows
# the hot-path table marks "next" carry that tag. The headline is the largest
# single-GPU workload.
WORKLOADS = [("tiny_decode", "C1"), ("gqa_decode", "C2"), ("spec_decode", "C3"),
             ("alibi_decode", "C4"), ("mqa_split", "C5"), ("mla_decode", "next"),
             ("prefill_causal", "next")]
HEADLINE = "alibi_decode"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None,
                    help="measure this workload alone (default: every workload, "
                         f"headline {HEADLINE})")
    ap.add_argument("--chunk-blocks", type=int, default=None)
    ap.add_argument("--config-steps", type=int, default=300,
                    help="timed steps of each non-headline workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=100)
    return ap.parse_args()


def peaks():
    """(HBM GB/s, dense fp16/bf16 tensor TFLOP/s burst, 'measured' | 'fallback').
    fp16 and bf16 run at the same nominal tensor rate, so the measured bf16
    GEMM figure serves fp16 with ratio 1."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_TFLOPS)), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_TFLOPS, "fallback"


# Device sources of each attention kernel: an ncu figure stays valid while
# these files are unchanged.
KERNEL_SOURCES = {
    "mma_decode_kernel": ["pa_decode_mma.cuh", "pa_decode_mma.cu"],
    "fma_decode_kernel": ["pa_decode_fma.cuh"],
    "tc_decode_kernel": ["pa_decode_tc.cuh", "pa_decode_tc.cu"],
    "wide_decode_kernel": ["pa_decode_wide.cuh", "pa_decode_wide.cu", "pa_decode_mma.cuh"],
    "pf_attn_kernel": ["pa_prefill_tc.cuh", "pa_prefill_tc.cu", "pa_decode_tc.cuh"],
    "pf_pair_kernel": ["pa_prefill_pair.cuh", "pa_prefill_pair.cu", "pa_prefill_tc.cuh",
                       "pa_decode_tc.cuh"],
}
COMMON_SOURCES = ["pa_device.cuh", "pa_warp_pipe.cuh"]


def kernel_sources_sha(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_206_gb300", "csrc")
    for f in COMMON_SOURCES + KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "pa.h"), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    sources are unchanged since it was taken (else None)."""
    p = os.path.join(ROOT, "profiles", f"{kernel}.{workload}.txt")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m_sha = re.search(r"^source_sha:\s*(\S+)", text, re.M)
    m_b = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    if not (m_sha and m_b) or m_sha.group(1) != kernel_sources_sha(kernel):
        return None
    return float(m_b.group(1))


def dominant_kernel(cfg, shared_kv=False):
    """The attention kernel pa_forward picks for this configuration (shared_kv:
    value_cache is key_cache)."""
    rows = (cfg.num_heads // cfg.kv_heads) * max(1, cfg.max_seqlen_q)
    if rows > 64 and cfg.head_size_k == cfg.head_size_v and cfg.head_size_k in (64, 128):
        return "pf_pair_kernel" if rows > 128 else "pf_attn_kernel"
    hk, hv = cfg.head_size_k, cfg.head_size_v
    wide = shared_kv and ((hk, hv) == (576, 512) or (hk == hv and hk in (256, 512)))
    if 8 < rows <= 16 and wide:
        return "wide_decode_kernel"
    if rows > 8:
        return "tc_decode_kernel"
    mma = (cfg.head_size_k == cfg.head_size_v and cfg.head_size_k in (64, 128, 256, 512)) or \
        (cfg.head_size_k, cfg.head_size_v) == (576, 512)
    return "mma_decode_kernel" if rows >= 2 and mma else "fma_decode_kernel"


def launches_per_step(n_combine):
    """Kernels one pa_forward launches: the attention kernel, plus the combine
    kernel (its programmatic dependent) when the plan has split tiles."""
    return 1 + (1 if n_combine else 0)


class ClockSampler:
    """nvidia-smi clock and throttle samples while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in (self.out or "").splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        # samples taken while the GPU was busy: the upper half of the clock readings
        busy = sorted(sm)[len(sm) // 2:]
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def workload(name, rank, chunk):
    from paged_kv_cache_206_gb300 import workloads as W
    w = W.NAMED[name](seed=rank)
    if chunk is not None:
        w.chunk_blocks = chunk
    return w


def flush_l2(flush):
    """Evict the L2 (129 MB) before a timed step: write the 512 MB buffer, then
    read half of it back, so that the write's dirty lines are written back to
    HBM here rather than inside the next timed step."""
    import torch
    flush.zero_()
    flush[: flush.numel() // 2].view(torch.float32).sum()


def time_device(fn, steps, warmup, flush, stream):
    """Per-step CUDA-event times (ms) of fn() on `stream`, L2 flushed before each step."""
    import torch
    for _ in range(warmup):
        flush_l2(flush)
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush_l2(flush)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def percentiles(xs):
    """median, p10 and p90 of a list (nearest rank)."""
    ys = sorted(xs)
    pick = lambda f: ys[min(len(ys) - 1, max(0, int(round(f * (len(ys) - 1)))))]
    return {"median": pick(0.5), "p10": pick(0.1), "p90": pick(0.9)}


def cpu_baseline(w, max_seconds=10.0):
    """The oracle on this machine's cores, on the whole batch or a prefix of it
    sized to stay within about max_seconds."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    order = list(range(w.batch))
    # estimate from one sequence, then take as many sequences as fit
    t0 = time.perf_counter()
    _, used = oracle.attention(w, subset=order[:1], threads=cores)
    one = time.perf_counter() - t0
    per_seq = max(one / max(1, min(used, 1)), 1e-4)
    n = max(1, min(w.batch, int(max_seconds * min(cores, w.batch) / per_seq)))
    sub = order[:n]
    t0 = time.perf_counter()
    _, used = oracle.attention(w, subset=sub, threads=cores)
    dt = time.perf_counter() - t0
    per = w.head_size_k + (0 if w.shared_kv else w.head_size_v)
    kv = int(w.context_lens[sub].astype(np.int64).sum()) * w.kv_heads * per * 2
    return {"value": kv / dt / 1e9, "unit": UNIT, "cores": int(used), "kind": "oracle",
            "seconds": dt,
            "sample": f"{n} of {w.batch} sequences ({kv / 1e9:.3f} GB of KV), fp64 C oracle, "
                      f"OpenMP over (sequence, kv head)"}


def reduce_over_ranks(maxes, sums, world, device):
    """Whole-job figures of independent replicas: the slowest rank's times
    (max) and the bytes and tokens of all ranks (sum). One collective each; the
    data path itself has none."""
    if world <= 1:
        return list(maxes), list(sums)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(maxes), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor(list(sums), device=device, dtype=torch.float64)
    dist.all_reduce(u)
    return t.tolist(), u.tolist()


def reference_sample(w, nseq: int, nkv: int):
    """The first nseq sequences of w restricted to its first nkv kv heads (and
    their query heads): a smaller batch of the same shapes and values, the
    reference arm's per-step sample."""
    import dataclasses
    G = w.num_heads // w.kv_heads
    H = nkv * G
    nq = int(w.q_seqlens[:nseq].sum())
    mask = w.mask
    if mask is not None and mask.ndim == 3:  # MASK_TYPE_NORM: one mask per sequence
        mask = np.ascontiguousarray(mask[:nseq])
    # (a shared-KV workload's value_cache already holds the first hv dims of K)
    kc = np.ascontiguousarray(w.key_cache[:, :, :nkv])
    vc = np.ascontiguousarray(w.value_cache[:, :, :nkv])
    return dataclasses.replace(
        w, num_heads=H, kv_heads=nkv, context_lens=w.context_lens[:nseq].copy(),
        q_seqlens=w.q_seqlens[:nseq].copy(), block_tables=w.block_tables[:nseq].copy(),
        query=np.ascontiguousarray(w.query[:nq, :H]), key_cache=kc, value_cache=vc, mask=mask,
        alibi_slopes=None if w.alibi_slopes is None else w.alibi_slopes[:H].copy())


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    name = args.workload or HEADLINE
    w = workload(name, 0, args.chunk_blocks)
    cores = len(os.sched_getaffinity(0))
    # Bounded sample per step, sized so that the whole run (warm-up and timed
    # steps) takes about REF_BUDGET_S, at most 0.5 s a step: the first nseq
    # sequences with the first nkv kv heads. The oracle works on (sequence, kv
    # head) units, one thread each; one unit is the smallest sample.
    unit = reference_sample(w, 1, 1)
    t0 = time.perf_counter()
    oracle.attention(unit, threads=1)
    one = max(time.perf_counter() - t0, 1e-5)
    per_step = min(0.5, REF_BUDGET_S / max(1, args.steps + args.warmup))
    units = max(1, int(per_step * cores / one))
    nseq = min(w.batch, units)
    nkv = min(w.kv_heads, max(1, units // nseq))
    smp = reference_sample(w, nseq, nkv)
    kv = smp.kv_bytes()
    used = 1
    for _ in range(args.warmup):
        _, used = oracle.attention(smp, threads=cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _, used = oracle.attention(smp, threads=cores)
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    value = kv / dt / 1e9
    sample = (f"{nseq} of {w.batch} sequences x {nkv} of {w.kv_heads} kv heads per step, "
              f"fp64 C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": name, "sample_sequences": nseq, "sample_kv_heads": nkv,
                   "batch": w.batch},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": int(used), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def read_peak(dev, stream):
    """HBM read bandwidth of this GPU: pa_hbm_read_probe over 2 GiB (more than
    L2 holds), best mean over the grid shapes tried."""
    import torch
    import paged_kv_cache_206_gb300 as pa
    buf = torch.empty(READ_PROBE_BYTES, dtype=torch.uint8, device=dev)
    buf.fill_(1)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    best = None
    for ctas in (1, 2, 4):
        for _ in range(3):
            pa.hbm_read_probe(buf, ctas, sink, stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(20)]
        for a, b in ev:
            a.record(stream)
            pa.hbm_read_probe(buf, ctas, sink, stream)
            b.record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        gbs = READ_PROBE_BYTES / (ms * 1e-3) / 1e9
        if best is None or gbs > best["gbs"]:
            best = {"gbs": gbs, "ctas_per_sm": ctas, "ms": ms}
    del buf
    torch.cuda.empty_cache()  # give the 2 GiB back before the workloads
    return {"value": best["gbs"], "unit": "GB/s", "bytes": READ_PROBE_BYTES,
            "ctas_per_sm": best["ctas_per_sm"],
            "how": "pa_hbm_read_probe: 256-bit loads (L1 bypassed, L2 evict-first), "
                   "512 threads a CTA, 8 loads in flight a thread; best of 1/2/4 CTAs per SM, "
                   "mean of 20 launches each"}


def measure(name, args, steps, dev, stream, flush, rank, peaks_, read_gbs, cpu_seconds):
    """Every figure of one workload: the device step, its roofline, the end-to-end
    step from host buffers (with its stages timed) and the oracle on the host."""
    import torch
    import paged_kv_cache_206_gb300 as pa

    w = workload(name, rank, args.chunk_blocks)
    db = pa.DeviceBatch(w, device=dev)
    ql_host = None if np.all(w.q_seqlens == 1) else w.q_seqlens
    plan_reps = 50
    t0 = time.perf_counter()
    for _ in range(plan_reps):
        pa.pa_plan(db.cfg, w.context_lens, ql_host)
    plan_us = (time.perf_counter() - t0) / plan_reps * 1e6
    kv_bytes, qo_bytes = w.kv_bytes(), w.qo_bytes()
    n_comb = db.plan.combine.shape[0]
    n_items = db.plan.work.shape[0]
    launches = launches_per_step(n_comb)

    times = time_device(lambda: db.forward(stream), steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    st, bits = db.status(stream)
    if st != pa.PA_OK:
        raise RuntimeError(f"{name}: kernel status {pa.status_string(st)} ({bits})")
    # the attention kernel alone (the roofline's kernel): the same launch
    # without the combine list, which launches no combine kernel; without
    # split tiles the step is that one launch
    if n_comb:
        def attention_only():
            pa.pa_forward(db.cfg, db.query, db.key_cache, db.value_cache, db.block_tables,
                          db.context_lens, db.q_seqlens, db.mask, db.alibi_slopes, db.work,
                          None, db.workspace, db.out, stream)
        kernel_ms = statistics.mean(time_device(attention_only, steps, 5, flush, stream))
        db.forward(stream)
    else:
        kernel_ms = statistics.mean(times)

    # end to end through the C ABI with host buffers: GraphStep replays one
    # graph per step (copy in, device plan, attention storing the output into
    # pinned host memory; the host waits); HostStep plans on the host and
    # launches directly; the graph's
    # stages are also run directly with events between them
    def fill(st_):
        st_.query.copy_(torch.from_numpy(np.ascontiguousarray(w.query)))
        st_.block_tables.copy_(torch.from_numpy(np.ascontiguousarray(w.block_tables)))
        st_.context_lens.copy_(torch.from_numpy(np.ascontiguousarray(w.context_lens)))
        if st_.q_seqlens is not None:
            st_.q_seqlens.copy_(torch.from_numpy(np.ascontiguousarray(w.q_seqlens)))
        return st_

    gs = fill(pa.GraphStep(db.cfg, db.key_cache, db.value_cache, w.total_q, mask=db.mask,
                           alibi_slopes=db.alibi_slopes))
    hs = fill(pa.HostStep(db.cfg, db.key_cache, db.value_cache, w.total_q, mask=db.mask,
                          alibi_slopes=db.alibi_slopes))

    def time_host(fn, n):
        for _ in range(min(5, n)):
            fn()
        out = []
        for _ in range(n):
            flush_l2(flush)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            out.append(time.perf_counter() - t0)
        return out

    e2e_t = time_host(gs.run, args.e2e_steps)
    host_t = time_host(lambda: hs.run(stream), args.e2e_steps)
    # the stages queue up behind the L2 flush (the step's stream waits for the
    # flush's), so the events measure the GPU's time on each stage rather
    # than the host's time to enqueue the next one
    stage_ms = [[] for _ in range(4)]
    for _ in range(max(1, args.e2e_steps // 2)):
        torch.cuda.synchronize()
        flush_l2(flush)
        gs.stream.wait_stream(torch.cuda.current_stream(dev))
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        gs.run_stages(ev)
        for k in range(4):
            stage_ms[k].append(ev[k].elapsed_time(ev[k + 1]))
    if e2e_t:
        for what, s_ in (("graph", gs.status()), ("host-planned", hs.status(stream))):
            if s_[0] != pa.PA_OK:
                raise RuntimeError(f"{name}: e2e {what} status {pa.status_string(s_[0])} ({s_[1]})")
        db.forward(stream)
        ref_out = db.out.cpu()
        if not (torch.equal(gs.out, ref_out) and torch.equal(hs.out, ref_out)):
            raise RuntimeError(f"{name}: end-to-end output differs from the device-resident run")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    ms = statistics.mean(times)
    e2e_s = statistics.mean(e2e_t) if e2e_t else float("nan")
    host_s = statistics.mean(host_t) if host_t else float("nan")
    (ms_all, e2e_all, host_all), (kv_all, q_all) = reduce_over_ranks(
        [ms, e2e_s, host_s], [kv_bytes, w.total_q], world, dev)
    peak, tpeak, peak_kind = peaks_
    value = kv_all / (ms_all * 1e-3) / 1e9
    flops = w.attn_flops()
    tensor_bound = flops / (kv_bytes + qo_bytes) > tpeak * 1e3 / peak
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": flops / (kernel_ms * 1e-3) / 1e12, "peak": tpeak,
                "unit": "TFLOP/s", "flops": flops,
                "bytes": "2*(hk+hv) flop per (query row, visible key), algorithmic"}
        roof["frac"] = roof["achieved"] / roof["peak"]
    else:
        achieved = (kv_bytes + qo_bytes) / (kernel_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "bytes": "KV + Q + O per launch (algorithmic)", "frac": achieved / peak,
                "read_peak": read_gbs, "frac_read": achieved / read_gbs if read_gbs else None}
    kernel = dominant_kernel(db.cfg, w.shared_kv)
    base = None
    if not args.no_cpu_baseline and world == 1:
        base = cpu_baseline(w, cpu_seconds)
    stages = [statistics.mean(x) * 1e3 for x in stage_ms]
    res = {
        "value": value, "unit": UNIT, "ms_per_step": ms_all, "steps": steps,
        "step_ms": dict(percentiles(times), mean=ms),
        "pct_of_nominal_8tbs": 100.0 * value / NOMINAL_HBM_GBS,
        "query_tokens_per_s": q_all / (ms_all * 1e-3),
        "config": {
            "workload": name, "batch": w.batch, "num_heads": w.num_heads,
            "kv_heads": w.kv_heads, "head_size_k": w.head_size_k, "head_size_v": w.head_size_v,
            "block_size": w.block_size, "q_per_seq": w.max_seqlen_q, "mask_type": w.mask_type,
            "shared_kv": w.shared_kv, "kv_bytes": kv_bytes, "qo_bytes": qo_bytes,
            "items": n_items, "combines": n_comb, "chunk_blocks": db.cfg.chunk_blocks,
            "split_merge": "combine kernel" if n_comb else "none",
            "l2": "flushed before every step, outside the events: 512 MB written, then 256 MB "
                  "read back",
            "plan_us": plan_us},
        "roofline": dict(roof, traffic=ncu_traffic(kernel, name), peak_kind=peak_kind,
                         kernel=kernel, kernel_ms=kernel_ms, launches_per_step=launches),
        "e2e": None if not e2e_t else {
            "value": kv_all / e2e_all / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": int(gs.h2d_bytes),
            "d2h_bytes_per_step": int(gs.out.numel() * gs.out.element_size()),
            "ms_per_step": e2e_all * 1e3,
            "path": "GraphStep: one graph replay per step (device plan reading the lengths "
                    "from pinned host memory, beside the copy of the inputs; attention and "
                    "combine storing an output of at most 4 MiB straight into pinned host "
                    "memory, a larger one into device memory, then copied), host waits",
            "out_to_host": "kernels write pinned memory" if gs.d_out is None else "copy",
            "breakdown_us": {"h2d_copy": stages[0], "plan_device": stages[1],
                             "attention": stages[2], "d2h_copy": stages[3],
                             "how": "the graph's stages enqueued one after another (the whole "
                                    "arena copied first, no overlap) on its stream behind the L2 "
                                    "flush, CUDA events between them"},
            "host_planned": {"value": kv_all / host_all / 1e9, "ms_per_step": host_all * 1e3,
                             "h2d_bytes_per_step": int(hs.last_h2d_bytes),
                             "path": "HostStep: pa_plan on the host, direct launches"}},
        "gpu_launches": steps * launches,
        "cpu_baseline": base,
    }
    del gs, hs, db
    torch.cuda.empty_cache()
    return res


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import paged_kv_cache_206_gb300 as pa
    from paged_kv_cache_206_gb300 import build_lib
    if rank == 0 or world == 1:
        build_lib.build()
    if world > 1:
        dist.barrier()
    pa.load_library()

    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) == 36:
        gpu_id = "GPU-" + gpu_id
    peaks_ = peaks()
    names = [args.workload] if args.workload else [n for n, _ in WORKLOADS]
    headline = args.workload or HEADLINE
    rows = dict(WORKLOADS)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    results = {}
    with ClockSampler(gpu_id) as clk:
        rp = read_peak(dev, stream)
        for n in names:
            steps = args.steps if n == headline else min(args.steps, args.config_steps)
            results[n] = measure(n, args, steps, dev, stream, flush, rank, peaks_, rp["value"],
                                 10.0 if n == headline else 3.0)
            results[n]["row"] = rows.get(n, "-")
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    h = results[headline]
    line = {
        "metric": METRIC,
        "value": h["value"],
        "unit": UNIT,
        "n_gpus": world,
        "steps": h["steps"],
        "warmup": args.warmup,
        "ms_per_step": h["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": dict(h["config"], parallelism=f"replica x{world}" if world > 1 else "single"),
        "step_ms": h["step_ms"],
        "query_tokens_per_s": h["query_tokens_per_s"],
        "pct_of_nominal_8tbs": h["pct_of_nominal_8tbs"],
        "roofline": h["roofline"],
        "e2e": h["e2e"],
        "gpu_launches": h["gpu_launches"],
        "clocks": clk.summary(),
        "cpu_baseline": h["cpu_baseline"],
        "hbm_read_peak": rp,
        "configs": results,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
