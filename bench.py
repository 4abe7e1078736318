"""Benchmark: paged-KV GQA split-decode on one GB300 (or N independent replicas).

One step = one pass of the whole hot path over one synthetic batch: the plan
refresh (planner kernel), the split-KV decode kernel and the merge kernel, all
through the C ABI, captured in a CUDA graph and replayed.  The headline workload
is the largest single-GPU batch, the Large skewed batch (512 seqs, context
lognormal(median 2048, sigma 1.2) in [16, 65536], Hq/Hkv 64/8, D 128, page 128,
bf16); its ~8.6 GB of KV per step is far larger than the 129 MB L2, so no flush
is needed between steps.

Prints one JSON line (rank 0).  `value` is the algorithmic KV-read bandwidth,
sum_r S_r * Hkv * D * 2 (K and V) * elem_bytes per step, over the measured step
time; `us_per_decode_call` is the pa_decode call (split + merge, the refresh
excluded; a graph of K calls) and `us_per_refresh` the refresh alone.  With the
default workload the same line also carries the Large batch with an fp8 cache
(`large_fp8`), the skewed agentic batch over --seeds seeds (`skewed_seeds`:
median / p10 fraction of the measured HBM copy peak, and the uniform-split
plan's time over the proportional plan's on the same kernel, L2 flushed before
every step) and three multi-token verify batches (`verify`: the skewed fp8
batch x 3 tokens, 16 x 16384 keys x 3 tokens in fp8, and MTP verify; L2
flushed).  `--sweep all` adds one line per configuration (L2 flushed before
every step) and a summary over the skewed batch's seeds.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--workload NAME] [--seeds S] [--sweep]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_decode_split_gb300 import binding, workloads as wl  # noqa: E402

METRIC = "paged-decode KV-read GB/s vs ~8 TB/s HBM roofline; µs per decode call"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "large_bf16"
DESCRIBE = {
    "tiny": "tiny decode: 4 seqs, ctx {17,64,200,1000}, Hq/Hkv 8/2, D 64, page 16, bf16",
    "uniform": "uniform decode: 32 seqs x 8192 ctx, Hq/Hkv 32/4, D 128, page 16, bf16",
    "skewed": "skewed agentic decode: 32 seqs, ctx lognormal(4096, 1.5) in [64,131072], "
              "Hq/Hkv 32/4, D 128, page 16, fp8-e4m3 KV (scale 0.05), budget 296, cap 256",
    "mtp_verify": "MTP verify: 8 req x 3 tok at 16384 ctx, Hq/Hkv 6/1, D 256, page 64, bf16, "
                  "8 padding rows",
    "mixed_prompt": "mixed: 7 decodes at 16384 + one 100-token prompt, Hq/Hkv 12/2, D 256, "
                    "page 64, bf16, 21 padding rows",
    "large_bf16": "large skewed: 512 seqs, ctx lognormal(2048, 1.2) in [16,65536], Hq/Hkv 64/8, "
                  "D 128, page 128, bf16",
    "large_fp8": "large skewed: 512 seqs, ctx lognormal(2048, 1.2) in [16,65536], Hq/Hkv 64/8, "
                 "D 128, page 128, fp8-e4m3 KV",
    "large_bf16_quarter": "the first 128 requests of the large skewed batch (Hq/Hkv 64/8, D 128, "
                          "page 128, bf16): a profiling-sized case",
    "uniform_w1024": "uniform decode under a 1024-key sliding window",
    "skewed_w4096": "skewed agentic decode under a 4096-key sliding window",
    "uniform_k5": "uniform decode with K in the grouped layout [nb, Hkv, D/16, 16, 16]",
    "skewed_k5": "skewed agentic decode with K in the grouped layout [nb, Hkv, D/16, 16, 16]",
    "uniform_d512": "uniform decode: 16 seqs x 8192 ctx, Hq/Hkv 32/4, D 512, page 16, bf16",
    "uniform_d1024": "uniform decode: 16 seqs x 8192 ctx, Hq/Hkv 32/4, D 1024, page 16, bf16",
    "uniform_n64_h8": "uniform decode: 64 seqs x 4096 ctx, Hq/Hkv 64/8, D 128, page 16, bf16",
    "skewed_mtp3": "MTP verify on the skewed agentic batch: 32 seqs x 3 query tokens, ctx "
                   "lognormal(4096, 1.5) in [64,131072], Hq/Hkv 32/4, D 128, page 16, fp8-e4m3 KV "
                   "(scale 0.05), budget 296, cap 256",
    "skewed_d1024": "skewed agentic decode: 32 seqs, ctx lognormal(4096, 1.5) in [64,131072], "
                    "Hq/Hkv 16/2, D 1024, page 16, fp8-e4m3 KV (scale 0.05), K grouped, "
                    "budget 296, cap 256",
}
for _kv, _kvd in (("fp8", "fp8-e4m3 KV (scale 0.05)"), ("bf16", "bf16 KV")):
    for _t in (1, 2, 3, 4):
        DESCRIBE[f"rows_{_kv}_t{_t}"] = (f"verify rows: 16 seqs x {_t} query token(s) at 16384 ctx, "
                                         f"Hq/Hkv 32/4, D 128, page 16, {_kvd}")
SPLIT_SOURCES = ["pa_split.cuh", "pa_split_cfg.h", "pa_device.cuh", "pa_fused.cuh"]
L2_BYTES = 129 * 1024 * 1024


# ------------------------------------------------------------------ helpers

def split_kernel_sha() -> str:
    h = hashlib.sha256()
    for f in SPLIT_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_decode_split_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


def ncu_traffic(workload: str):
    """DRAM bytes per split-kernel launch from the committed ncu summary, or None
    when absent or taken on a different version of the kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except OSError:
        return None
    e = d.get(workload)
    if not e or e.get("kernel_sha") != split_kernel_sha():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples SM clock, max clock and clock-event reasons through NVML (read
    only) on a background thread while active."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: torch.device):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self._stop = threading.Event()
        self._active = threading.Event()
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            props = torch.cuda.get_device_properties(device)
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._h = nv, h
        except OSError:
            return
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def _run(self):
        nv, h = self._nvml, self._h
        c, r = ctypes.c_uint(), ctypes.c_ulonglong()
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if self._active.wait(0.05):
                if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) == 0:
                    self.samples.append(c.value)
                if fn(h, ctypes.byref(r)) == 0:
                    self.reasons |= r.value
                time.sleep(0.0005)

    def start(self):
        self._active.set()

    def stop(self):
        self._active.clear()

    def close(self) -> dict | None:
        self._stop.set()
        if self._nvml is None:
            return None
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples),
                "reasons": [n for b, n in self.REASONS.items() if self.reasons & b]}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest value of x over all ranks (harness timing only)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# -------------------------------------------------------------- CPU oracle

def oracle_sample(w, max_seconds: float = 20.0):
    """Times the fp64 oracle on a bounded sample of the workload's requests: a
    first request calibrates its speed, then requests are taken in order while
    the estimated cost stays under half the budget.
    Returns (KV GB/s, seconds, cores, description)."""
    import oracle

    per_req = w.kv_bytes_per_request().tolist()
    n = len(per_req)
    sub = wl.subset(w, [0])
    t0 = time.perf_counter()
    _run_oracle(sub)
    dt = time.perf_counter() - t0
    per_byte = dt / max(1, per_req[0])
    picks, total = [0], per_req[0]
    for r in range(1, n):
        if per_byte * (total + per_req[r]) >= max_seconds / 2:
            break
        picks.append(r)
        total += per_req[r]
    sub = wl.subset(w, picks)
    t0 = time.perf_counter()
    _run_oracle(sub)
    dt = time.perf_counter() - t0
    desc = (f"{len(picks)} of {n} requests ({sub.kv_bytes() / 1e6:.1f} MB of "
            f"{w.kv_bytes() / 1e6:.1f} MB KV), all query rows and heads, fp64")
    return sub.kv_bytes() / dt / 1e9, dt, oracle.num_threads(), desc


def _run_oracle(w):
    import numpy as np
    import oracle
    q = w.q.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    if w.kv_dtype == "fp8":
        k = w.k_cache.cpu().contiguous().numpy()
        v = w.v_cache.cpu().contiguous().numpy()
    else:
        k = w.k_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        v = w.v_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    code = {"bf16": oracle.BF16, "fp16": oracle.FP16, "fp8": oracle.FP8_E4M3}[w.kv_dtype]
    qc = oracle.FP16 if w.q.dtype == torch.float16 else oracle.BF16
    cu = None if w.cu_query_lens is None else w.cu_query_lens.cpu().numpy()
    return oracle.decode(q, qc, k, v, code, w.k_scale, w.v_scale, w.block_tables.cpu().numpy(),
                         w.context_lens.cpu().numpy(), cu, w.scale, window=w.window)


# ------------------------------------------------------------ GPU timings

def _graph(fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _replay_ms(g, dev) -> float:
    """Device time of one replay of g (events on the replaying stream)."""
    cur = torch.cuda.current_stream(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(cur)
    g.replay()
    t1.record(cur)
    torch.cuda.synchronize(dev)
    return t0.elapsed_time(t1)


def _step_fns(w, kind, out, fused=None):
    """(plan, refresh, decode) for a Workload, or for a SparseWorkload: there the
    refresh is the block selection followed by the plan refresh from the
    selected lengths, and the decode runs over the sparse block table."""
    if isinstance(w, wl.SparseWorkload):
        sw, b = w, w.base
        plan = binding.Plan(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim,
                            max_partitions=sw.max_partitions, budget=b.budget or 0, kind=kind,
                            device=b.q.device)
        if fused is not None:
            plan.set_fused_merge(fused)
        sel = torch.empty((b.num_seqs, sw.sel_stride), dtype=torch.int32, device=b.q.device)
        sl = torch.empty(b.num_seqs, dtype=torch.int32, device=b.q.device)

        def refresh():
            binding.sparse_select(sw.scores, b.context_lens, b.block_tables, b.block_size,
                                  sw.top_k, sw.init_blocks, sw.local_blocks, sel, sl)
            plan.refresh(sl)

        def decode():
            plan.decode(b.q, b.k_cache, b.v_cache, sel, sl, None, b.scale, b.k_scale, b.v_scale,
                        out=out)
        return plan, refresh, decode
    plan = binding.plan_for(w, kind)
    if fused is not None:
        plan.set_fused_merge(fused)
    return (plan, lambda: plan.refresh(w.context_lens, w.cu_query_lens),
            lambda: binding.decode_workload(plan, w, out=out))


def time_native(w, steps: int, warmup: int, kind=binding.PROPORTIONAL, flush: bool = False,
                sampler: ClockSampler | None = None, world: int = 1, fused=None):
    """Graph-replayed timing of K steps, as a serving engine replays its decode
    graphs.  A step is refresh + decode (planner, split, merge kernels).

    Pass 1 (the number): the K steps captured in one CUDA graph with nothing
    else inside, timed by an event pair around its replay.  With flush=True
    every step is preceded by an L2 flush (write a 2xL2 buffer, then read
    another, so that no dirty line is written back inside the timed kernels),
    and the replay time of a graph of the K flushes alone is subtracted.
    Pass 2: the same with K pa_decode calls alone (the plan refreshed once
    before): the decode call time.  Pass 3 (the breakdown): the steps with
    per-step events that the library records around the split kernel; their
    median (an event pair between kernels costs the launch overlap, so this
    errs long).

    A SparseWorkload's step is selection + refresh + decode over the selection.
    fused: None keeps the plan's default merge; True / False force the merge
    inside the split kernel / the separate merge kernel.

    Returns dict(step_ms, call_ms, split_ms, split_all) and the plan."""
    q = w.base.q if isinstance(w, wl.SparseWorkload) else w.q
    dev = q.device
    out = torch.empty_like(q)
    plan, refresh_fn, decode_fn = _step_fns(w, kind, out, fused)
    fa = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    fb = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    sink = torch.empty(steps, dtype=torch.float32, device=dev) if flush else None
    ev = lambda: torch.cuda.Event(enable_timing=True)
    splits = [(ev(), ev()) for _ in range(steps)]

    def flush_l2(i):
        fa.zero_()
        torch.sum(fb, dim=0, out=sink[i])

    def body(events: bool, work: bool = True, refresh: bool = True):
        for i in range(steps):
            if flush:
                flush_l2(i)
            if not work:
                continue
            if events:
                plan.set_split_events(*splits[i])
            if refresh:
                refresh_fn()
            decode_fn()
        plan.set_split_events(None, None)

    cur = torch.cuda.current_stream(dev)
    for _ in range(max(warmup, 3)):
        refresh_fn()
        decode_fn()
    for a, b in splits:  # materialise the CUDA events before handing them to the ABI
        a.record(cur)
        b.record(cur)
    torch.cuda.synchronize(dev)
    g_plain = _graph(lambda: body(False))
    g_call = _graph(lambda: body(False, refresh=False))
    g_flush = _graph(lambda: body(False, work=False)) if flush else None
    g_events = _graph(lambda: body(True))
    g_plain.replay()
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
    total = _replay_ms(g_plain, dev)
    if sampler:
        sampler.stop()
    barrier(world)
    g_call.replay()
    torch.cuda.synchronize(dev)
    calls = _replay_ms(g_call, dev)
    if g_flush is not None:
        fl = _replay_ms(g_flush, dev)
        total -= fl
        calls -= fl
    g_events.replay()
    torch.cuda.synchronize(dev)
    split_all = [a.elapsed_time(b) for a, b in splits]
    del g_plain, g_call, g_flush, g_events
    return {"step_ms": total / steps, "call_ms": calls / steps,
            "split_ms": statistics.median(split_all), "split_all": split_all}, plan


def time_refresh(w, reps: int = 100) -> float:
    """µs per plan refresh (for a SparseWorkload: selection + refresh): a graph
    of `reps` of them, replayed."""
    q = w.base.q if isinstance(w, wl.SparseWorkload) else w.q
    plan, refresh_fn, _ = _step_fns(w, binding.PROPORTIONAL, None)
    refresh_fn()
    torch.cuda.synchronize()
    g = _graph(lambda: [refresh_fn() for _ in range(reps)])
    g.replay()
    ms = _replay_ms(g, q.device)
    del g
    return ms * 1e3 / reps


def time_e2e(w, steps: int, warmup: int, kv_resident: bool = False):
    """Same metric through the public API with host-resident inputs: every step
    copies the step's inputs from pinned host memory, runs refresh + decode, and
    reads the output back.  kv_resident=False copies everything -- q, K, V,
    block tables, lengths (and cu); kv_resident=True copies what changes from
    one decode step to the next in a serving engine -- q, block tables, lengths
    (and cu) -- while the paged KV cache stays in HBM.  As a serving engine
    overlaps the next batch's upload with the current batch's attention, the
    copies of step i+1 run on a copy stream into the other of two device buffer
    sets while step i decodes; the timed region spans the first upload to the
    last read-back."""
    dev = w.q.device
    names = ["q", "block_tables", "context_lens"]
    if not kv_resident:
        names[1:1] = ["k_cache", "v_cache"]
    if w.cu_query_lens is not None:
        names.append("cu_query_lens")
    host = {n: getattr(w, n).cpu().pin_memory() for n in names}
    sets = [{n: torch.empty_like(getattr(w, n)) for n in names} for _ in range(2)]
    wds = [wl.Workload(**{**w.__dict__, **d}) for d in sets]
    outs = [torch.empty_like(w.q) for _ in range(2)]
    out_h = torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory()
    plan = binding.plan_for(w)
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    uploaded = [ev(), ev()]   # set k holds a step's inputs
    consumed = [ev(), ev()]   # set k's last decode is done with its inputs

    def upload(i):
        k = i % 2
        copy.wait_event(consumed[k])
        with torch.cuda.stream(copy):
            for n in names:
                sets[k][n].copy_(host[n], non_blocking=True)
        uploaded[k].record(copy)

    def compute(i):
        k = i % 2
        comp.wait_event(uploaded[k])
        plan.refresh(wds[k].context_lens, wds[k].cu_query_lens)
        binding.decode_workload(plan, wds[k], out=outs[k])
        consumed[k].record(comp)
        out_h.copy_(outs[k], non_blocking=True)

    def run(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute(i)

    for k in range(2):
        consumed[k].record(comp)
    run(max(warmup, 3))
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    copy.wait_event(t0)
    run(steps)
    t1.record(comp)  # after the last read-back; every upload precedes a compute it waits for
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / steps
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    del host, sets, wds, outs
    return ms, h2d, d2h


def workload_dtype(w) -> str:
    return "fp8_e4m3 KV / fp16 MMA, fp32 accumulate" if w.kv_dtype == "fp8" else \
        f"{w.kv_dtype} MMA, fp32 accumulate"


# ------------------------------------------------------------------ arms

def plan_ab(w, steps: int, warmup: int, flush: bool, peak: float) -> dict:
    """The proportional and the uniform-split plan on the same kernel and batch:
    decode call and split kernel times, and their fractions of the copy peak."""
    kv = w.kv_bytes()
    tp, _ = time_native(w, steps, warmup, flush=flush)
    tu, _ = time_native(w, steps, warmup, kind=binding.UNIFORM, flush=flush)
    gbs = lambda ms: kv / (ms * 1e-3) / 1e9
    return {"kv_bytes": kv,
            "us_per_decode_call": round(tp["call_ms"] * 1e3, 2),
            "split_us": round(tp["split_ms"] * 1e3, 2),
            "call_gbs": round(gbs(tp["call_ms"]), 1),
            "call_frac_of_measured": round(gbs(tp["call_ms"]) / peak, 4),
            "split_frac_of_measured": round(gbs(tp["split_ms"]) / peak, 4),
            "uniform_us_per_decode_call": round(tu["call_ms"] * 1e3, 2),
            "uniform_split_us": round(tu["split_ms"] * 1e3, 2),
            "uniform_over_proportional_call": round(tu["call_ms"] / tp["call_ms"], 3),
            "uniform_over_proportional_split": round(tu["split_ms"] / tp["split_ms"], 3)}


def skewed_seeds(dev, seeds: int, steps: int, warmup: int, peak: float) -> dict:
    """The skewed agentic batch over seeds 0..seeds-1 (each a fresh length draw,
    cache and page order), both plans on the same kernel, L2 flushed before
    every step: medians and tails of the fractions of the copy peak and of the
    uniform plan's time over the proportional plan's."""
    rows = []
    for seed in range(seeds):
        w = wl.skewed(seed, dev)
        r = plan_ab(w, steps, warmup, True, peak)
        r["seed"] = seed
        r["max_over_min"] = round(w.meta["max_over_min"], 1)
        rows.append(r)
        del w
        torch.cuda.empty_cache()
    col = lambda k: [r[k] for r in rows]
    stat = lambda xs: {"median": _pct(xs, 0.5), "p10": _pct(xs, 0.1), "min": min(xs),
                       "max": max(xs)}
    return {"workload": DESCRIBE["skewed"], "seeds": seeds,
            "l2": "flushed before every step (write a 2xL2 buffer, read another)",
            "max_over_min": stat(col("max_over_min")),
            "call_frac_of_measured": stat(col("call_frac_of_measured")),
            "split_frac_of_measured": stat(col("split_frac_of_measured")),
            "us_per_decode_call": stat(col("us_per_decode_call")),
            "uniform_over_proportional_call": stat(col("uniform_over_proportional_call")),
            "uniform_over_proportional_split": stat(col("uniform_over_proportional_split")),
            "per_seed": [{k: r[k] for k in ("seed", "max_over_min", "us_per_decode_call",
                                            "uniform_us_per_decode_call",
                                            "call_frac_of_measured")} for r in rows]}


def run_native(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    if args.sweep_only:
        if rank == 0:
            sweep(args)
        return
    if args.profile_run:
        profile_run(args, dev)
        return
    t_start = time.perf_counter()
    w = wl.CONFIGS[args.workload](0, dev)
    kv_bytes = w.kv_bytes()
    sampler = ClockSampler(dev) if rank == 0 else None
    t, plan = time_native(w, args.steps, args.warmup, sampler=sampler, world=world)
    ms = max_over_ranks(t["step_ms"], world)
    info = plan.info()
    clocks = sampler.close() if sampler else None
    tu, _ = time_native(w, args.steps, args.warmup, kind=binding.UNIFORM)
    refresh_us = time_refresh(w)
    e2e_ms, h2d, d2h = time_e2e(w, args.steps, args.warmup)
    e2e_ms = max_over_ranks(e2e_ms, world)
    res_ms, res_h2d, res_d2h = time_e2e(w, args.steps, args.warmup, kv_resident=True)
    res_ms = max_over_ranks(res_ms, world)
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_kind = "measured" if peak else "fallback"
    peak = peak or 6800.0
    split_ms = t["split_ms"]
    achieved = kv_bytes / (split_ms * 1e-3) / 1e9
    traffic = ncu_traffic(args.workload)
    line = {
        "metric": METRIC, "value": round(world * kv_bytes / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "us_per_decode_call": round(t["call_ms"] * 1e3, 2),
        "decode_call_gbs": round(kv_bytes / (t["call_ms"] * 1e-3) / 1e9, 1),
        "us_per_refresh": round(refresh_us, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": workload_dtype(w), "data": "synthetic (seeded N(0,1) q/K/V, random page order)",
        "config": {"workload": DESCRIBE[args.workload], "name": args.workload,
                   "kv_bytes_per_step": kv_bytes, "plan": "proportional",
                   "budget": info["budget"], "capacity": info["capacity"],
                   "max_partitions": info["max_partitions"],
                   "step": "plan refresh + pa_decode (split-KV kernel + merge kernel)",
                   "l2": "inputs larger than L2 (no flush)" if kv_bytes > L2_BYTES
                   else "not flushed: inputs fit in L2",
                   "timing": "K steps captured once in a CUDA graph and replayed; decode "
                             "calls alone likewise; split time: median of per-step events "
                             "in a third replay",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "pa::split_kernel", "split_us_per_launch": round(split_ms * 1e3, 2),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel_sha": split_kernel_sha()},
        "plan_ab": {"proportional_us_per_step": round(ms * 1e3, 2),
                    "uniform_us_per_step": round(tu["step_ms"] * 1e3, 2),
                    "proportional_split_us": round(split_ms * 1e3, 2),
                    "uniform_split_us": round(tu["split_ms"] * 1e3, 2)},
        "e2e": {"value": round(world * kv_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "inputs": "q, K and V caches, block tables, lengths uploaded every step"},
        "e2e_kv_resident": {"value": round(world * kv_bytes / (res_ms * 1e-3) / 1e9, 1),
                            "unit": UNIT, "h2d_bytes_per_step": res_h2d,
                            "d2h_bytes_per_step": res_d2h, "ms_per_step": round(res_ms, 4),
                            "inputs": "q, block tables, lengths uploaded every step; the paged "
                                      "KV cache stays in HBM"},
        "gpu_launches": (1 + plan.kernels_per_decode()) * args.steps,
        "merge": "fused into the split kernel" if plan.fused_merge else "separate merge kernel",
        "clocks": clocks,
    }
    del w, plan
    torch.cuda.empty_cache()
    if args.workload == DEFAULT_WORKLOAD and rank == 0 and not args.no_extra:
        wf = wl.CONFIGS["large_fp8"](0, dev)
        line["large_fp8"] = {"workload": DESCRIBE["large_fp8"],
                             **plan_ab(wf, args.steps, args.warmup, False, peak)}
        del wf
        torch.cuda.empty_cache()
        if args.seeds > 0:
            line["skewed_seeds"] = skewed_seeds(dev, args.seeds, min(args.steps, 50),
                                                args.warmup, peak)
        # multi-token verify rows (speculative decoding): the fp8 skewed batch x
        # 3 tokens and 16 x 16384 keys x 3 tokens (tensor-memory consumer), and
        # MTP verify (bf16, D 256), both plans, L2 flushed before every step
        line["verify"] = {}
        for name in ("skewed_mtp3", "rows_fp8_t3", "mtp_verify"):
            wv = wl.CONFIGS[name](0, dev)
            line["verify"][name] = {"workload": DESCRIBE[name],
                                    **plan_ab(wv, min(args.steps, 50), args.warmup, True, peak)}
            del wv
            torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        w = wl.CONFIGS[args.workload](0, dev)
        gbs, secs, cores, desc = oracle_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": UNIT, "cores": cores,
                                "kind": "oracle", "sample": desc, "seconds": round(secs, 2)}
        del w
    line["wall_s"] = round(time.perf_counter() - t_start, 1)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if args.sweep and rank == 0:
        sweep(args)


def profile_run(args, dev):
    """For profilers: W + K plain (eager) steps of the workload -- refresh and
    decode, three kernel launches each -- with nothing else on the GPU; the
    first W are the warm-up to skip (ncu -s 3W for every kernel, -s W for one)."""
    w = wl.CONFIGS[args.workload](0, dev)
    plan = binding.plan_for(w)
    out = torch.empty_like(w.q)
    for _ in range(args.warmup + args.steps):
        plan.refresh(w.context_lens, w.cu_query_lens)
        binding.decode_workload(plan, w, out=out)
    torch.cuda.synchronize(dev)
    print(json.dumps({"profile_run": args.workload, "steps": args.steps, "warmup": args.warmup,
                      "kv_bytes_per_step": w.kv_bytes(), "errors": plan.read_errors()}),
          flush=True)


def _fusable(w) -> bool:
    """Whether a workload's plan can take the fused merge: head dim at most
    256, and every request's query rows (tokens x GQA group) in one work item
    of at most 32 rows."""
    b = w.base if isinstance(w, wl.SparseWorkload) else w
    g = b.num_q_heads // b.num_kv_heads
    if b.head_dim > 256 or g > 32:
        return False
    if b.cu_query_lens is None:
        return True
    cu = b.cu_query_lens.cpu()
    return int((cu[1:] - cu[:-1]).max()) * g <= 32


def _pct(xs, q):
    xs = sorted(xs)
    return xs[min(len(xs) - 1, int(round(q * (len(xs) - 1))))]


def sweep(args):
    """One line per configuration (and skewed seed): proportional vs uniform
    plan on the same kernel, L2 flushed before every step, graph-replayed;
    then a summary line over the skewed seeds (median, p90)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    names = (list(wl.CONFIGS) + list(wl.SPARSE_CONFIGS) if args.sweep == "all"
             else args.sweep.split(","))
    peak = measured_peaks().get("hbm_gbs", 6800.0)
    skew = []
    for name in names:
        seeds = range(args.seeds) if name == "skewed" else [0]
        for seed in seeds:
            w = (wl.SPARSE_CONFIGS[name] if name in wl.SPARSE_CONFIGS else wl.CONFIGS[name])(
                seed, dev)
            kv = w.kv_bytes()
            lens = (w.selected_tokens() if isinstance(w, wl.SparseWorkload)
                    else w.context_lens).tolist()
            res = {"sweep": name, "seed": seed, "kv_bytes": kv,
                   "max_over_min": round(max(lens) / max(1, min(lens)), 1)}
            for kind, tag in ((binding.PROPORTIONAL, "proportional"),
                              (binding.UNIFORM, "uniform")):
                t, plan = time_native(w, args.steps, args.warmup, kind=kind, flush=True)
                _, red = plan.download()
                res[tag] = {"us_per_step": round(t["step_ms"] * 1e3, 2),
                            "us_per_decode_call": round(t["call_ms"] * 1e3, 2),
                            "split_us": round(t["split_ms"] * 1e3, 2),
                            "call_gbs": round(kv / (t["call_ms"] * 1e-3) / 1e9, 1),
                            "split_gbs": round(kv / (t["split_ms"] * 1e-3) / 1e9, 1),
                            "split_frac_of_measured": round(kv / (t["split_ms"] * 1e-3) / 1e9 / peak, 4),
                            "call_frac_of_measured": round(kv / (t["call_ms"] * 1e-3) / 1e9 / peak, 4),
                            "split_frac_of_8tbs": round(kv / (t["split_ms"] * 1e-3) / 8e12, 4),
                            "tasks": int(red[:, 1].sum()), "max_parts": int(red[:, 1].max())}
            res["refresh_us"] = round(time_refresh(w), 2)
            if _fusable(w):  # A/B: the same plan with the merge fused into the split kernel
                t, _ = time_native(w, args.steps, args.warmup, flush=True, fused=True)
                res["fused_merge_us_per_decode_call"] = round(t["call_ms"] * 1e3, 2)
                res["merge_kernel_us_per_decode_call"] = res["proportional"]["us_per_decode_call"]
            print(json.dumps(res), flush=True)
            if name == "skewed":
                skew.append(res)
            del w
            torch.cuda.empty_cache()
    if skew:
        sp = [r["proportional"]["split_us"] for r in skew]
        cp = [r["proportional"]["us_per_decode_call"] for r in skew]
        fr = [r["proportional"]["split_frac_of_measured"] for r in skew]
        fc = [r["proportional"]["call_frac_of_measured"] for r in skew]
        su = [r["uniform"]["split_us"] / r["proportional"]["split_us"] for r in skew]
        mm = [r["max_over_min"] for r in skew]
        print(json.dumps({"sweep": "skewed_summary", "seeds": len(skew),
                          "max_over_min": {"min": min(mm), "median": _pct(mm, 0.5), "max": max(mm)},
                          "split_us": {"median": _pct(sp, 0.5), "p90": _pct(sp, 0.9)},
                          "decode_call_us": {"median": _pct(cp, 0.5), "p90": _pct(cp, 0.9)},
                          "split_frac_of_measured": {"median": _pct(fr, 0.5), "p10": _pct(fr, 0.1),
                                                     "min": min(fr)},
                          "decode_call_frac_of_measured": {"median": _pct(fc, 0.5),
                                                           "p10": _pct(fc, 0.1), "min": min(fc)},
                          "uniform_over_proportional_split": {"median": round(_pct(su, 0.5), 2),
                                                              "min": round(min(su), 2)}}),
              flush=True)


def run_reference(args, world, rank, local):
    """The fp64 CPU oracle as the reference arm, on this workload's config,
    metric and unit; each step a bounded sample of the workload."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    # the inputs are drawn where they are drawn for the native arm (the same
    # seeded batch); only the sampled request is copied to the host and timed
    gen = torch.device("cuda", local) if torch.cuda.is_available() else "cpu"
    w = wl.CONFIGS[args.workload](0, gen)
    lens = w.context_lens.tolist()
    # one request per step (the first), all its query rows and heads
    sub = wl.subset(w, [0])
    for _ in range(args.warmup):
        _run_oracle(sub)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _run_oracle(sub)
    dt = (time.perf_counter() - t0) / args.steps
    gbs = sub.kv_bytes() / dt / 1e9
    desc = (f"1 of {len(lens)} requests per step ({sub.kv_bytes() / 1e6:.1f} MB of "
            f"{w.kv_bytes() / 1e6:.1f} MB KV), all query rows and heads, fp64")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": DESCRIBE[args.workload], "name": args.workload},
            "cpu_baseline": {"value": round(gbs, 4), "unit": UNIT, "kind": "oracle",
                             "cores": oracle.num_threads(), "sample": desc},
            "e2e": {"value": round(gbs, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=list(wl.CONFIGS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--sweep", default="", help="'all' or comma list: extra per-config lines")
    ap.add_argument("--seeds", type=int, default=20, help="skewed seeds in the sweep")
    ap.add_argument("--sweep-only", action="store_true",
                    help="print the --sweep lines only (no headline line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0,
                    help="bound on the oracle's timed sample (cpu_baseline)")
    ap.add_argument("--profile-run", action="store_true",
                    help="W + K plain steps of the workload for a profiler (no timing)")
    ap.add_argument("--no-extra", action="store_true",
                    help="headline workload only (no large_fp8 / skewed_seeds / verify keys)")
    args = ap.parse_args(argv)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_native(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
