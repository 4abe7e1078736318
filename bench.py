"""Benchmark: paged-KV GQA split-decode on one GB300 (or N independent replicas).

One step = one pass of the whole hot path over one synthetic batch: the plan
refresh (planner kernel), the split-KV decode kernel and the merge kernel, all
through the C ABI.  The headline workload is the uniform decode batch (32 seqs x
8192 context, Hq/Hkv 32/4, D 128, page 16, bf16); its 537 MB of KV per step is
larger than the 129 MB L2, so no flush is needed between steps.

Prints one JSON line (rank 0).  `value` is the algorithmic KV-read bandwidth,
sum_r S_r * Hkv * D * 2 (K and V) * elem_bytes per step, over the measured time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--workload NAME] [--sweep]
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
DEFAULT_WORKLOAD = "uniform"
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
}
SPLIT_SOURCES = ["pa_split.cuh", "pa_device.cuh"]
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
    """Times the fp64 oracle on a bounded sample of the workload's requests.
    Returns (KV GB/s, seconds, cores, description)."""
    import numpy as np
    import oracle

    lens = w.context_lens.cpu().tolist()
    # grow the sample one request at a time until its estimated cost reaches
    # ~1/4 of the budget (first call calibrates the per-byte speed)
    order = list(range(len(lens)))
    picks = [order[0]]
    sub = wl.subset(w, picks)
    t0 = time.perf_counter()
    _run_oracle(sub)
    dt = time.perf_counter() - t0
    per_byte = dt / max(1, sub.kv_bytes())
    target = max_seconds / 2
    i = 1
    while i < len(order) and per_byte * wl.subset(w, picks + [order[i]]).kv_bytes() < target:
        picks.append(order[i])
        i += 1
    sub = wl.subset(w, picks)
    t0 = time.perf_counter()
    _run_oracle(sub)
    dt = time.perf_counter() - t0
    desc = (f"{len(picks)} of {len(lens)} requests ({sub.kv_bytes() / 1e6:.1f} MB of "
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
                         w.context_lens.cpu().numpy(), cu, w.scale)


# ------------------------------------------------------------ GPU timings

def time_native(w, steps: int, warmup: int, kind=binding.PROPORTIONAL, flush: bool = False,
                sampler: ClockSampler | None = None, world: int = 1, graph: bool = True):
    """Device-timed steps (refresh + decode).  The K steps are captured once into
    a CUDA graph (refresh and decode are capturable: no allocation, no host
    synchronisation) and replayed, as a serving engine replays its decode
    graphs; each step records its own event pair around the split kernel.
    With flush=True every step is preceded by an L2-flushing write and timed
    by its own event pair.  Returns (ms/step, split-kernel ms per launch, plan)."""
    dev = w.q.device
    plan = binding.plan_for(w, kind)
    out = torch.empty_like(w.q)
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    ev = lambda: torch.cuda.Event(enable_timing=True)
    pairs = [(ev(), ev()) for _ in range(steps)]
    step_ev = [(ev(), ev()) for _ in range(steps)] if flush else None

    def step():
        plan.refresh(w.context_lens, w.cu_query_lens)
        binding.decode_workload(plan, w, out=out)

    def body(stream):
        for i, (a, b) in enumerate(pairs):
            if flush:
                flush_buf.zero_()
                step_ev[i][0].record(stream)
            plan.set_split_events(a, b)
            step()
            if flush:
                step_ev[i][1].record(stream)

    cur = torch.cuda.current_stream(dev)
    for _ in range(max(warmup, 3)):
        step()
    for a, b in pairs:  # materialise the CUDA events before handing them to the ABI
        a.record(cur)
        b.record(cur)
    if step_ev:
        for a, b in step_ev:
            a.record(cur)
            b.record(cur)
    torch.cuda.synchronize(dev)
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body(torch.cuda.current_stream(dev))
        plan.set_split_events(None, None)
        g.replay()  # warm replay
        torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0, t1 = ev(), ev()
    if sampler:
        sampler.start()
    t0.record(cur)
    if g is not None:
        g.replay()
    else:
        body(cur)
    t1.record(cur)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.stop()
    barrier(world)
    plan.set_split_events(None, None)
    if flush:
        ms = statistics.median(a.elapsed_time(b) for a, b in step_ev)
    else:
        ms = t0.elapsed_time(t1) / steps
    split_ms = statistics.mean(a.elapsed_time(b) for a, b in pairs)
    del g
    return ms, split_ms, plan


def time_e2e(w, steps: int, warmup: int):
    """Same metric through the public API with host-resident inputs: every step
    copies q, K, V, block tables, lengths (and cu) from pinned host memory, runs
    refresh + decode, and reads the output back."""
    dev = w.q.device
    names = ["q", "k_cache", "v_cache", "block_tables", "context_lens"]
    if w.cu_query_lens is not None:
        names.append("cu_query_lens")
    host = {n: getattr(w, n).cpu().pin_memory() for n in names}
    devt = {n: torch.empty_like(getattr(w, n)) for n in names}
    out_h = torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory()
    wd = wl.Workload(**{**w.__dict__, **devt})
    plan = binding.plan_for(w)
    out = torch.empty_like(w.q)
    stream = torch.cuda.current_stream(dev)

    def step():
        for n in names:
            devt[n].copy_(host[n], non_blocking=True)
        plan.refresh(wd.context_lens, wd.cu_query_lens)
        binding.decode_workload(plan, wd, out=out)
        out_h.copy_(out, non_blocking=True)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / steps
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    return ms, h2d, d2h


def workload_dtype(w) -> str:
    return "fp8_e4m3 KV / fp16 MMA, fp32 accumulate" if w.kv_dtype == "fp8" else \
        f"{w.kv_dtype} MMA, fp32 accumulate"


# ------------------------------------------------------------------ arms

def run_native(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    w = wl.CONFIGS[args.workload](0, dev)
    kv_bytes = w.kv_bytes()
    sampler = ClockSampler(dev) if rank == 0 else None
    ms, split_ms, plan = time_native(w, args.steps, args.warmup, sampler=sampler, world=world)
    ms = max_over_ranks(ms, world)
    info = plan.info()
    clocks = sampler.close() if sampler else None
    ms_u, split_u, plan_u = time_native(w, args.steps, args.warmup, kind=binding.UNIFORM)
    e2e_ms, h2d, d2h = time_e2e(w, args.steps, args.warmup)
    e2e_ms = max_over_ranks(e2e_ms, world)
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_kind = "measured" if peak else "fallback"
    peak = peak or 6800.0
    achieved = kv_bytes / (split_ms * 1e-3) / 1e9
    traffic = ncu_traffic(args.workload)
    line = {
        "metric": METRIC, "value": round(world * kv_bytes / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "us_per_decode_call": round(ms * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": workload_dtype(w), "data": "synthetic (seeded N(0,1) q/K/V, random page order)",
        "config": {"workload": DESCRIBE[args.workload], "name": args.workload,
                   "kv_bytes_per_step": kv_bytes, "plan": "proportional",
                   "budget": info["budget"], "capacity": info["capacity"],
                   "max_partitions": info["max_partitions"],
                   "l2": "inputs larger than L2 (no flush)" if kv_bytes > L2_BYTES
                   else "not flushed: inputs fit in L2",
                   "timing": "K steps captured once in a CUDA graph and replayed",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "pa::split_kernel", "split_us_per_launch": round(split_ms * 1e3, 2),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel_sha": split_kernel_sha()},
        "plan_ab": {"proportional_us": round(ms * 1e3, 2), "uniform_us": round(ms_u * 1e3, 2)},
        "e2e": {"value": round(world * kv_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, secs, cores, desc = oracle_sample(w)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": UNIT, "cores": cores,
                                "kind": "oracle", "sample": desc, "seconds": round(secs, 2)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if args.sweep and rank == 0:
        sweep(args)


def sweep(args):
    """One line per configuration: proportional vs uniform plan on the same kernel,
    L2 flushed between steps, median step time."""
    dev = torch.device("cuda", torch.cuda.current_device())
    names = [n for n in wl.CONFIGS if n != "tiny"] if args.sweep == "all" else \
        args.sweep.split(",")
    for name in names:
        seeds = range(args.seeds) if name == "skewed" else [0]
        for seed in seeds:
            w = wl.CONFIGS[name](seed, dev)
            kv = w.kv_bytes()
            res = {"sweep": name, "seed": seed, "kv_bytes": kv,
                   "max_over_min": round(max(w.context_lens.tolist()) /
                                         max(1, min(w.context_lens.tolist())), 1)}
            for kind, tag in ((binding.PROPORTIONAL, "proportional"),
                              (binding.UNIFORM, "uniform")):
                ms, split_ms, plan = time_native(w, args.steps, args.warmup, kind=kind, flush=True,
                                                 graph=False)
                _, red = plan.download()
                res[tag] = {"us_per_call": round(ms * 1e3, 2),
                            "split_us": round(split_ms * 1e3, 2),
                            "kv_gbs": round(kv / (ms * 1e-3) / 1e9, 1),
                            "split_gbs": round(kv / (split_ms * 1e-3) / 1e9, 1),
                            "frac_of_measured": round(kv / (split_ms * 1e-3) / 1e9 /
                                                      measured_peaks().get("hbm_gbs", 6800.0), 4),
                            "tasks": int(red[:, 1].sum()), "max_parts": int(red[:, 1].max())}
            # refresh alone: 100 refreshes captured in a graph, replayed
            plan = binding.plan_for(w)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            plan.refresh(w.context_lens, w.cu_query_lens)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(100):
                    plan.refresh(w.context_lens, w.cu_query_lens)
            g.replay()
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            res["refresh_us"] = round(a.elapsed_time(b) * 10, 2)
            del g
            print(json.dumps(res), flush=True)
            del w
            torch.cuda.empty_cache()


def run_reference(args, world, rank, local):
    """The fp64 CPU oracle as the reference arm, on this workload's config,
    metric and unit; each step a bounded sample of the workload."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = wl.CONFIGS[args.workload](0, "cpu")
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
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=list(wl.CONFIGS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--sweep", default="", help="'all' or comma list: extra per-config lines")
    ap.add_argument("--seeds", type=int, default=3, help="skewed seeds in the sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
