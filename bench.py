"""Benchmark: dense FP8 MQA logits on the 2048 x 32768, H=64, D=128 workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one mqa_logits call over the whole workload (clean fp32 logits,
rows [0, S_kv - S_q + i)).  Timing: W untimed warm-up steps, then K steps,
each timed with CUDA events on the launching stream, L2 flushed (a 256 MiB
write) before every step outside the events, a barrier and a device
synchronize around the timed loop, the max over ranks.  Prints one JSON line.

--impl reference times the CPU oracle (the plain double-precision reference in
oracle/) on a bounded row sample of the same workload on this host's cores.
Other workloads: the 2048 x 4096 and 8192 x 65536 dense calls, the paged decode
call, and the top-k key selection over 2048 x 32768 logits rows
(topk_2k_32k_k2048, reported in rows/s against the HBM roofline).
Under torchrun each rank runs the whole workload on its own GPU (the rows are
independent; no collective is on the data path) and rank 0 reports the
aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0   # nominal dense FP8 : BF16 tensor rate (4.5 : 2.25 PFLOP/s)
KERNEL_SOURCES = ["fp8_mqa_indexer_gb300/csrc/mqa_kernel.cuh", "fp8_mqa_indexer_gb300/csrc/ptx.cuh",
                  "fp8_mqa_indexer_gb300/csrc/launch.h"]
TOPK_SOURCES = ["fp8_mqa_indexer_gb300/csrc/mqa_topk.cu", "fp8_mqa_indexer_gb300/csrc/topk.h"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


FP8_PEAK_FILE = os.path.join(ROOT, "profiles", "fp8_peak.json")


def committed_fp8_peak():
    """The FP8 GEMM peak a default benchmark run measured on this machine's GB300
    (profiles/fp8_peak.json), for lines run without their own measurement."""
    if not os.path.exists(FP8_PEAK_FILE):
        return None
    with open(FP8_PEAK_FILE) as f:
        return json.load(f)


def fp8_roofline_peak(fp8, nominal_peak, peaks_src):
    """(peak, source): the live FP8 measurement, else the committed one, else
    the bf16 burst x 2."""
    if fp8:
        return fp8["burst_tflops"], "measured fp8 (cuBLAS e4m3 GEMM burst on this GPU)"
    rec = committed_fp8_peak()
    if rec:
        return rec["burst_tflops"], "measured fp8 (cuBLAS e4m3 GEMM burst, profiles/fp8_peak.json)"
    return nominal_peak, f"{peaks_src} bf16 burst x {FP8_PER_BF16} (nominal fp8:bf16)"


def recorded_traffic(workload: str, sources=KERNEL_SOURCES):
    """DRAM bytes per launch from a committed ncu capture, if the kernel is unchanged."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f).get(workload)
    if not rec or rec.get("kernel_hash") != kernel_hash(sources):
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def percentiles(times_ms):
    xs = sorted(times_ms)

    def q(f):
        k = (len(xs) - 1) * f
        lo, hi = int(k), min(int(k) + 1, len(xs) - 1)
        return xs[lo] + (xs[hi] - xs[lo]) * (k - lo)
    return {"median_ms": q(0.5), "p10_ms": q(0.1), "p90_ms": q(0.9)}


# Dense E4M3 tensor-core work per SM and SM clock: one 128 x 256 x 128 MMA
# unit (8.4 MFLOP) issues every 512 cycles when nothing else limits it (an
# MMA-only issue loop on this GPU); used for the fraction at the kernel's own
# clock.
FP8_FLOP_PER_SM_CLK = 16384


def measure_fp8_peak(torch, dev, seconds: float = 4.0, n: int = 8192):
    """Dense FP8 (E4M3 x E4M3, fp32 accumulate) GEMM rate of this GPU through
    cuBLAS (torch._scaled_mm, bf16 out) at n^3: best of 10 (burst) and back to
    back for `seconds` (sustained), with the SM clocks sampled meanwhile."""
    g = torch.Generator(device=dev).manual_seed(7)
    a = torch.randn((n, n), device=dev, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn((n, n), device=dev, generator=g).to(torch.float8_e4m3fn).t()
    one = torch.ones((), device=dev, dtype=torch.float32)

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

    flop = 2.0 * n ** 3
    for _ in range(3):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[0].strip() if vis else str(dev.index or 0))
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    iters = 0
    t0 = time.perf_counter()
    e0.record()
    while time.perf_counter() - t0 < seconds:
        for _ in range(20):
            mm()
        iters += 20
        torch.cuda.synchronize()
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    sustained = flop * iters / (e0.elapsed_time(e1) * 1e-3) / 1e12
    del a, b
    return {"burst_tflops": flop / (best * 1e-3) / 1e12, "sustained_tflops": sustained,
            "sustained_sm_mhz": clocks.get("sm_mhz"), "sustained_reasons": clocks.get("reasons"),
            "how": f"torch._scaled_mm e4m3 x e4m3 -> bf16, {n}^3 (2*n^3 FLOP): best of 10 (burst) "
                   f"and back to back for {seconds:.0f} s (sustained)"}


def pre_spin(torch):
    """A 0.2 ms one-thread spin on the timing stream right before the start
    event: the host issues the timed call while the GPU spins, so the event
    interval holds the call's device time and not the host's launch latency
    (that is part of the end-to-end figure).  It touches no memory, so the L2
    stays flushed."""
    torch.cuda._sleep(400_000)


def graph_timing(torch, call, out, calls: int = 5, samples: int = 40):
    """Timing in the manner of the PR #435 reproducer: one CUDA graph holding
    `calls` calls, each writing its own output buffer, replayed `samples`
    times; per-call time of every replay (CUDA events) -> median, p10, p90."""
    outs = [out] + [torch.empty_like(out) for _ in range(calls - 1)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for o in outs:
            call(o)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for o in outs:
            call(o)
    graph.replay()
    torch.cuda.synchronize()
    per_call = []
    for _ in range(samples):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        per_call.append(e0.elapsed_time(e1) / calls)
    del graph, outs
    r = percentiles(per_call)
    r.update({"calls_per_graph": calls, "samples": samples,
              "note": "no L2 flush between calls; each call writes its own output buffer"})
    return r


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def make_case(workload: str):
    from fp8_mqa_indexer_gb300 import workloads as wl
    if workload in wl.TOPK_CONFIGS:
        return wl.topk_config(workload)
    if workload in wl.FUSED_CONFIGS:
        return wl.fused_config(workload)[0]
    if workload in wl.PAGED_CONFIGS:
        return wl.paged_config(workload)
    if workload in wl.PAGED_MX_CONFIGS:
        return wl.paged_mx_config(workload)
    if workload in wl.MX_CONFIGS:
        return wl.mx_config(workload)
    if workload not in wl.DENSE_CONFIGS:
        raise SystemExit(f"unknown workload {workload!r}; known: "
                         f"{sorted(wl.DENSE_CONFIGS) + sorted(wl.PAGED_CONFIGS) + sorted(wl.PAGED_MX_CONFIGS) + sorted(wl.TOPK_CONFIGS) + sorted(wl.MX_CONFIGS)}")
    return wl.dense_config(workload)


def is_paged(workload: str) -> bool:
    from fp8_mqa_indexer_gb300 import workloads as wl
    return workload in wl.PAGED_CONFIGS or workload in wl.PAGED_MX_CONFIGS


def is_mx(workload: str) -> bool:
    from fp8_mqa_indexer_gb300 import workloads as wl
    return workload in wl.MX_CONFIGS


# The pages' MXFP8 timings ("[PR #435] ...", section "Performance": GB200, 152
# SMs, all-zero input, clean fp32 logits, CUDA-graph median per call), as
# TFLOP/s of this benchmark's metric (valid logits x 2 * H * D).
MX_PUBLISHED_US = {"mx_2k_32k_h64_d128_zeros": 412.0, "mx_8k_64k_h64_d128_zeros": 3022.2,
                   "mx4_2k_32k_h64_d128_zeros": 407.9, "mx4_8k_64k_h64_d128_zeros": 2968.9}


def bench_mx(args, mqa, torch, dev, stream):
    """MXFP8 or MXFP4 dense logits (block-scaled tcgen05 MMA); the shapes of
    the pages' MX timings."""
    from fp8_mqa_indexer_gb300 import workloads as wl
    case = wl.mx_config(args.workload)
    i = torch.arange(case.S_q, dtype=torch.int64)
    valid = int((case.k_end.to(torch.int64).clamp(max=case.S_kv)
                 - case.k_start.to(torch.int64).clamp(min=0)).clamp(min=0).sum())
    flops = valid * 2.0 * case.H * 128
    d = [t.to(dev) for t in (case.q, case.q_sf, case.kv, case.kv_sf, case.weights, case.k_start,
                             case.k_end)]
    out = torch.empty((case.S_q, case.ldo), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(o=out):
        mqa.mqa_logits_mx(*d, o, fp4=case.fp4)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[0].strip() if vis else "0")
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        pre_spin(torch)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    assert mqa.device_status() == 0
    times_ms = [a.elapsed_time(b) for a, b in ev]
    ms_per_step = sum(times_ms) / args.steps
    value = flops / (ms_per_step * 1e-3) / 1e12
    graph = None
    if not args.no_graph:
        graph = graph_timing(torch, step, out)
        graph["tflops_at_median"] = flops / (graph["median_ms"] * 1e-3) / 1e12

    host = [t.pin_memory() for t in (case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                     case.k_start, case.k_end)]
    host_out = torch.empty((case.S_q, case.ldo), dtype=torch.float32, pin_memory=True)

    def e2e_step():
        dd = [h.to(dev, non_blocking=True) for h in host]
        mqa.mqa_logits_mx(*dd, out, fp4=case.fp4)
        host_out.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb) / args.e2e_steps

    peaks, peaks_src = load_peaks()
    nominal_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    fp8 = None if args.no_fp8_peak else measure_fp8_peak(torch, dev)
    peak, peak_source = fp8_roofline_peak(fp8, nominal_peak, peaks_src)
    published = MX_PUBLISHED_US.get(args.workload)
    pub_tflops = flops / (published * 1e-6) / 1e12 if published else None
    if graph and pub_tflops:
        graph["vs_published_median"] = graph["tflops_at_median"] / pub_tflops
    line = {
        "metric": "MQA logits TFLOP/s (valid logits x 2*H*D)",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": value / pub_tflops if pub_tflops else None,
        "dtype": ("mxfp4 (e2m1 x e2m1" if case.fp4 else "mxfp8 (e4m3 x e4m3") +
                 ", ue8m0 block 32) -> f32", "data": "synthetic",
        "config": {"workload": args.workload, "S_q": case.S_q, "S_kv": case.S_kv, "H": case.H,
                   "D": 128, "valid_logits": valid, "clean": True,
                   "l2": "flushed (256 MiB write) before every timed step",
                   "baseline": (f"{published} us on GB200 (the pages' "
                                f"{'MXFP4' if case.fp4 else 'MXFP8'} figure, all-zero input, "
                                f"graph median) = {pub_tflops:.0f} TFLOP/s" if published else None)},
        **percentiles(times_ms),
        "graph_timing": graph,
        "roofline": {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s",
                     "frac": value / peak, "traffic": recorded_traffic(args.workload),
                     "peak_source": peak_source,
                     "peak_bf16x2": nominal_peak, "frac_bf16x2": value / nominal_peak},
        "fp8_peak": fp8,
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in host),
                "d2h_bytes_per_step": host_out.numel() * 4, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def is_topk(workload: str) -> bool:
    from fp8_mqa_indexer_gb300 import workloads as wl
    return workload in wl.TOPK_CONFIGS


def topk_oracle_sample(case, budget_s: float):
    """Time the oracle's top-k on evenly spread rows until ~budget_s of wall time."""
    import oracle
    import numpy as np
    oracle.build()
    cores = max(1, len(os.sched_getaffinity(0)))
    L = case.logits.numpy()
    ks, ke = case.k_start.numpy(), case.k_end.numpy()
    order = list(range(0, case.rows, max(1, case.rows // 256)))
    order += [r for r in range(case.rows) if r not in set(order)]
    done, t0, k = 0, time.perf_counter(), 0
    while k < len(order):
        batch = order[k:k + cores]
        k += len(batch)
        oracle.run_rows_parallel(
            lambda r: oracle.topk_indices(L, ks, ke, topk=case.topk, n_cols=case.n_cols,
                                          rows=(r, r + 1)), batch, threads=cores)
        done += len(batch)
        if time.perf_counter() - t0 >= budget_s:
            break
    wall = time.perf_counter() - t0
    return {"rows_per_s": done / wall, "cores": cores, "rows": done, "wall_s": wall}


def bench_topk(args, mqa, torch, dev, stream):
    """Top-k key selection over a logits matrix; an HBM-bound path."""
    from fp8_mqa_indexer_gb300 import workloads as wl
    case = wl.topk_config(args.workload)
    R = case.rows
    valid = int(case.valid_counts().sum())
    # algorithmic bytes: every in-range logit read once, the index matrix and the ranges
    alg_bytes = valid * 4 + R * case.topk * 4 + R * 8
    L = case.logits.to(dev)
    ks, ke = case.k_start.to(dev), case.k_end.to(dev)
    out = torch.empty((R, case.topk), dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(L_, ks_, ke_):
        mqa.mqa_topk_indices(L_, ks_, ke_, case.topk, out, S_kv=case.n_cols)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step(L, ks, ke)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[0].strip() if vis else "0")
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        pre_spin(torch)
        a.record(stream)
        step(L, ks, ke)
        b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    times_ms = [a.elapsed_time(b) for a, b in ev]
    ms_per_step = sum(times_ms) / args.steps

    host = {k: v.pin_memory() for k, v in dict(L=case.logits, ks=case.k_start, ke=case.k_end).items()}
    host_out = torch.empty((R, case.topk), dtype=torch.int32, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values())

    def e2e_step():
        d = {k: v.to(dev, non_blocking=True) for k, v in host.items()}
        step(d["L"], d["ks"], d["ke"])
        host_out.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb) / args.e2e_steps

    peaks, peaks_src = load_peaks()
    achieved = alg_bytes / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": "top-k key selection rows/s",
        "value": R / (ms_per_step * 1e-3), "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 -> i32", "data": "synthetic",
        "config": {"workload": args.workload, "rows": R, "n_cols": case.n_cols, "topk": case.topk,
                   "in_range_logits": valid,
                   "l2": "flushed (256 MiB write) before every timed step; the logits exceed L2",
                   "step": "mqa_topk_indices"},
        **percentiles(times_ms),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": recorded_traffic(args.workload, TOPK_SOURCES),
                     "algorithmic_bytes": alg_bytes, "peak_source": f"{peaks_src} HBM copy"},
        "e2e": {"value": R / (e2e_ms * 1e-3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": host_out.numel() * 4, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        info = topk_oracle_sample(case, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": info["rows_per_s"], "unit": "rows/s", "cores": info["cores"],
                                "kind": "oracle",
                                "sample": f"{info['rows']} of {R} rows ({info['wall_s']:.1f} s of "
                                          f"oracle time)" + (", throughput extrapolated"
                                                             if info["rows"] < R else "")}
    print(json.dumps(line), flush=True)
    return 0


def is_fused(workload: str) -> bool:
    from fp8_mqa_indexer_gb300 import workloads as wl
    return workload in wl.FUSED_CONFIGS


def fused_oracle_sample(case, topk: int, budget_s: float):
    """Time the oracle's logits and top-k, row by row, on evenly spread rows."""
    import oracle
    import numpy as np
    oracle.build()
    cores = max(1, len(os.sched_getaffinity(0)))
    order = list(range(0, case.S_q, max(1, case.S_q // 256)))
    order += [r for r in range(case.S_q) if r not in set(order)]

    def one(r):
        L = oracle.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                              case.k_end, clean=False, rows=(r, r + 1))
        return oracle.topk_indices(L, case.k_start[r:r + 1], case.k_end[r:r + 1], topk=topk,
                                   n_cols=case.S_kv)

    done, t0, k = 0, time.perf_counter(), 0
    while k < len(order):
        batch = order[k:k + cores]
        k += len(batch)
        oracle.run_rows_parallel(one, batch, threads=cores)
        done += len(batch)
        if time.perf_counter() - t0 >= budget_s:
            break
    wall = time.perf_counter() - t0
    return {"rows_per_s": done / wall, "cores": cores, "rows": done, "wall_s": wall}


def bench_fused(args, mqa, torch, dev, stream):
    """Fused logits + top-k (mqa_logits_topk) on the dense workload's inputs,
    with the unfused pipeline (mqa_logits, then mqa_topk_indices) timed beside
    it.  The roofline is the logits contraction over the whole call."""
    from fp8_mqa_indexer_gb300 import workloads as wl
    case, topk = wl.fused_config(args.workload)
    R = case.S_q
    valid = int(case.valid_counts().sum())
    flops = valid * 2.0 * case.H * case.D
    d = dict(q=case.q, kv=case.kv, s=case.kv_scale, w=case.weights, ks=case.k_start,
             ke=case.k_end)
    dd = {k: v.to(dev) for k, v in d.items()}
    out = torch.empty((R, topk), dtype=torch.int32, device=dev)
    ws = torch.empty(mqa.mqa_logits_topk_workspace_size(R, case.S_kv), dtype=torch.uint8,
                     device=dev)
    L = torch.empty((R, case.S_kv), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(x):
        mqa.mqa_logits_topk(x["q"], x["kv"], x["s"], x["w"], x["ks"], x["ke"], topk, out,
                            workspace=ws)

    def unfused(x):
        mqa.mqa_logits(x["q"], x["kv"], x["s"], x["w"], x["ks"], x["ke"], L, clean=False)
        mqa.mqa_topk_indices(L, x["ks"], x["ke"], topk, out)

    def timed(fn, n):
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            fn(dd)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            flush.zero_()
            pre_spin(torch)
            a.record(stream)
            fn(dd)
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[0].strip() if vis else "0")
    sampler.start()
    time.sleep(0.3)
    times_ms = timed(step, args.steps)
    clocks = sampler.stop()
    ms_per_step = sum(times_ms) / args.steps
    unfused_ms = sorted(timed(unfused, max(5, args.steps // 2)))
    unfused_med = unfused_ms[len(unfused_ms) // 2]

    host = {k: (v.view(torch.uint8) if v.dtype == torch.float8_e4m3fn else v).pin_memory()
            for k, v in d.items()}
    host_out = torch.empty((R, topk), dtype=torch.int32, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values())

    def e2e_step():
        x = {k: v.to(dev, non_blocking=True) for k, v in host.items()}
        step(x)
        host_out.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb) / args.e2e_steps

    peaks, peaks_src = load_peaks()
    fp8 = None if args.no_fp8_peak else measure_fp8_peak(torch, dev)
    peak, peak_src = fp8_roofline_peak(fp8, peaks["bf16_tflops"] * 2.0, peaks_src)
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    line = {
        "metric": "fused logits + top-k rows/s",
        "value": R / (ms_per_step * 1e-3), "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 -> i32", "data": "synthetic",
        "config": {"workload": args.workload, "S_q": R, "S_kv": case.S_kv, "H": case.H,
                   "D": case.D, "topk": topk, "valid_logits": valid,
                   "l2": "flushed (256 MiB write) before every timed step",
                   "step": "mqa_logits_topk (split, candidate logits of each row's tail, "
                           "threshold, candidate logits of the rest, selection)"},
        **percentiles(times_ms),
        "unfused_ms": unfused_med,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "algorithmic_flops": flops,
                     "scope": "the whole call (five kernels), not one kernel",
                     "peak_source": peak_src},
        "e2e": {"value": R / (e2e_ms * 1e-3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": host_out.numel() * 4, "ms_per_step": e2e_ms},
        "gpu_launches": 5 * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        info = fused_oracle_sample(case, topk, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": info["rows_per_s"], "unit": "rows/s", "cores": info["cores"],
                                "kind": "oracle",
                                "sample": f"{info['rows']} of {R} rows ({info['wall_s']:.1f} s of "
                                          f"oracle time), throughput extrapolated"}
    print(json.dumps(line), flush=True)
    return 0


def paged_oracle_sample(case, budget_s: float):
    """Time the oracle on whole sequences (both of their rows) for ~budget_s."""
    import oracle
    oracle.build()
    cores = max(1, len(os.sched_getaffinity(0)))
    counts = case.valid_counts()
    rows, flops = 0, 0.0
    t0 = time.perf_counter()
    b = 0
    while b < case.B:
        batch = list(range(b, min(case.B, b + cores)))
        b += len(batch)

        def one(seq):
            r0 = seq * case.next_n
            if hasattr(case, "q_sf"):   # MX keys
                return oracle.paged_mx_mqa_logits(case.q, case.q_sf, case.kv_cache, case.kv_sf,
                                                  case.weights, case.context_lens, case.block_table,
                                                  next_n=case.next_n, fp4=case.fp4, ldo=case.ldo,
                                                  rows=(r0, r0 + case.next_n))
            return oracle.paged_mqa_logits(case.q, case.kv_cache, case.kv_scales, case.weights,
                                           case.context_lens, case.block_table,
                                           next_n=case.next_n, ldo=case.ldo, clean=case.clean,
                                           rows=(r0, r0 + case.next_n))
        oracle.run_rows_parallel(one, batch, threads=cores)
        rows += len(batch) * case.next_n
        flops += float(sum(int(counts[r]) for s_ in batch
                           for r in range(s_ * case.next_n, (s_ + 1) * case.next_n))) * 2 * case.H * case.D
        if time.perf_counter() - t0 >= budget_s:
            break
    wall = time.perf_counter() - t0
    return {"tflops": flops / wall / 1e12, "cores": cores, "rows": rows, "wall_s": wall}


def bench_paged(args, mqa, torch, dev, stream):
    """Paged decode: schedule + logits per step; an HBM-bound path."""
    case = make_case(args.workload)
    valid = int(case.valid_counts().sum())
    flops = valid * 2.0 * case.H * case.D
    R = case.B * case.next_n
    ctx = case.context_lens.to(torch.int64)
    pages = ((ctx.clamp(min=0) + case.block_kv - 1) // case.block_kv)
    mx = hasattr(case, "q_sf")   # MX keys: a scale word per key slot, per query row and head
    # algorithmic bytes: every key of every context (its row of E4M3 or packed
    # E2M1 bytes + its fp32 scale or scale word) once, the query rows (and
    # their scale words), weights, block-table entries in use, and the output
    alg_bytes = (int(ctx.clamp(min=0).sum()) * (case.kv_cache.shape[2] + 4) + case.q.numel()
                 + (case.q_sf.numel() * 4 if mx else 0) + case.weights.numel() * 4
                 + int(pages.sum()) * 4 + case.B * 4 + R * case.ldo * 4)
    src = dict(q=case.q, kvc=case.kv_cache, sc=case.kv_sf if mx else case.kv_scales, w=case.weights,
               cl=case.context_lens, bt=case.block_table)
    if mx:
        src["qsf"] = case.q_sf
    dd = {k: v.to(dev) for k, v in src.items()}
    cl = dd["cl"]
    out = torch.empty((R, case.ldo), dtype=torch.float32, device=dev)
    meta = torch.empty((mqa.get_num_sms(dev) + 1, 2), dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def logits(d, o):
        if mx:
            mqa.paged_mqa_logits_mx(d["q"], d["qsf"], d["kvc"], d["sc"], d["w"], d["cl"], d["bt"],
                                    meta, o, next_n=case.next_n, fp4=case.fp4)
        else:
            mqa.paged_mqa_logits(d["q"], d["kvc"], d["sc"], d["w"], d["cl"], d["bt"], meta, o,
                                 next_n=case.next_n, clean=case.clean)

    def step(d):
        mqa.paged_mqa_logits_metadata(d["cl"], next_n=case.next_n, block_kv=case.block_kv, out=meta)
        logits(d, out)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step(dd)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[0].strip() if vis else "0")
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        pre_spin(torch)
        a.record(stream)
        step(dd)
        b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    assert mqa.device_status() == 0
    times_ms = [a.elapsed_time(b) for a, b in ev]
    ms_per_step = sum(times_ms) / args.steps
    # the dominant kernel alone (the schedule computed once, as the pages'
    # reproducer does outside its timing), for the roofline
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in kev:
        flush.zero_()
        pre_spin(torch)
        a.record(stream)
        logits(dd, out)
        b.record(stream)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    kernel_ms = sum(a.elapsed_time(b) for a, b in kev) / args.steps

    host = {k: v.pin_memory() for k, v in src.items()}
    host_out = torch.empty((R, case.ldo), dtype=torch.float32, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values())

    def e2e_step():
        d = {k: v.to(dev, non_blocking=True) for k, v in host.items()}
        step(d)
        host_out.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb) / args.e2e_steps

    graph = None
    if not args.no_graph:
        def call(o):
            mqa.paged_mqa_logits_metadata(cl, next_n=case.next_n, block_kv=case.block_kv, out=meta)
            logits(dd, o)
        graph = graph_timing(torch, call, out)
        graph["gbs_at_median"] = alg_bytes / (graph["median_ms"] * 1e-3) / 1e9
    assert mqa.device_status() == 0

    peaks, peaks_src = load_peaks()
    achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
    line = {
        "metric": "MQA logits TFLOP/s (valid logits x 2*H*D)",
        "value": flops / (ms_per_step * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (("mxfp4 (e2m1 x e2m1" if case.fp4 else "mxfp8 (e4m3 x e4m3") +
                  ", ue8m0 block 32) -> f32") if mx else "e4m3 x e4m3 -> f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": case.B, "next_n": case.next_n, "H": case.H,
                   "D": case.D, "block_kv": case.block_kv, "num_blocks": case.num_blocks,
                   "ldo": case.ldo, "valid_logits": valid, "clean": case.clean,
                   "l2": "flushed (256 MiB write) before every timed step; the pool exceeds L2",
                   "step": "paged_mqa_logits_metadata + " +
                           ("paged_mqa_logits_mx" if mx else "paged_mqa_logits")},
        **percentiles(times_ms),
        "graph_timing": graph,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "kernel_ms": kernel_ms,
                     "kernel": ("paged_mqa_logits_mx" if mx else "paged_mqa_logits") +
                               " alone (event mean over the timed steps, L2 flushed); the step's "
                               "value includes the schedule kernel",
                     "step_gbs": alg_bytes / (ms_per_step * 1e-3) / 1e9,
                     "traffic": recorded_traffic(args.workload),
                     "algorithmic_bytes": alg_bytes, "peak_source": f"{peaks_src} HBM copy"},
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": host_out.numel() * 4,
                "ms_per_step": e2e_ms},
        "gpu_launches": 2 * args.steps,
        "kernel_only_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        info = paged_oracle_sample(case, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": info["tflops"], "unit": "TFLOP/s", "cores": info["cores"],
                                "kind": "oracle",
                                "sample": f"{info['rows']} of {R} rows ({info['wall_s']:.1f} s of "
                                          f"oracle time), throughput extrapolated"}
    print(json.dumps(line), flush=True)
    return 0


def oracle_sample(case, budget_s: float, max_rows: int = 4096):
    """Time the oracle on evenly spread rows until ~budget_s of wall time."""
    import oracle
    oracle.build()
    cores = max(1, len(os.sched_getaffinity(0)))
    stride_rows = list(range(0, case.S_q, max(1, case.S_q // 256)))
    order = stride_rows + [r for r in range(case.S_q) if r not in set(stride_rows)]
    counts = case.valid_counts()
    done_rows, flops = 0, 0.0
    t0 = time.perf_counter()
    k = 0
    while k < len(order) and done_rows < max_rows:
        batch = order[k:k + cores]
        k += len(batch)

        def one(r):
            if hasattr(case, "q_sf"):   # MXFP8 input
                return oracle.mx_mqa_logits(case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                            case.k_start, case.k_end, fp4=case.fp4, ldo=case.ldo,
                                            rows=(r, r + 1))
            return oracle.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                     case.k_end, ldo=case.ldo, clean=case.clean,
                                     compressed=case.compressed, rows=(r, r + 1))
        oracle.run_rows_parallel(one, batch, threads=cores)
        done_rows += len(batch)
        flops += float(sum(int(counts[r]) for r in batch)) * 2 * case.H * case.D
        if time.perf_counter() - t0 >= budget_s:
            break
    wall = time.perf_counter() - t0
    return {"tflops": flops / wall / 1e12, "cores": cores, "rows": done_rows, "wall_s": wall,
            "flops": flops}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    if is_topk(args.workload):
        return run_reference_topk(args)
    if is_fused(args.workload):
        return run_reference_fused(args)
    case = make_case(args.workload)
    valid = int(case.valid_counts().sum())
    flops_full = valid * 2.0 * case.H * case.D
    per_step = []
    info = None
    paged = is_paged(args.workload)
    for _ in range(args.warmup):
        if paged:
            paged_oracle_sample(case, budget_s=0.5)
        else:
            oracle_sample(case, budget_s=0.5, max_rows=8)
    budget = args.ref_budget or max(1.0, min(6.0, 90.0 / max(1, args.steps)))
    for _ in range(args.steps):
        info = paged_oracle_sample(case, budget_s=budget) if paged else oracle_sample(case, budget_s=budget)
        per_step.append(info["tflops"])
    value = statistics.median(per_step)
    ms_per_step = flops_full / (value * 1e12) * 1e3
    line = {
        "impl": "reference", "metric": "MQA logits TFLOP/s (valid logits x 2*H*D)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (exact e4m3 decode)",
        "data": "synthetic",
        "config": ({"workload": args.workload, "B": case.B, "next_n": case.next_n, "H": case.H,
                    "D": case.D, "valid_logits": valid, "clean": case.clean} if paged else
                   {"workload": args.workload, "S_q": case.S_q, "S_kv": case.S_kv, "H": case.H,
                    "D": case.D, "valid_logits": valid, "clean": case.clean}),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": info["cores"], "kind": "oracle",
                         "sample": f"{info['rows']} of {case.B * case.next_n if paged else case.S_q} rows per step, "
                                   f"extrapolated to the full workload ({info['wall_s']:.1f} s)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_fused(args):
    from fp8_mqa_indexer_gb300 import workloads as wl
    case, topk = wl.fused_config(args.workload)
    for _ in range(args.warmup):
        fused_oracle_sample(case, topk, budget_s=0.3)
    budget = args.ref_budget or max(1.0, min(6.0, 90.0 / max(1, args.steps)))
    per_step, info = [], None
    for _ in range(args.steps):
        info = fused_oracle_sample(case, topk, budget_s=budget)
        per_step.append(info["rows_per_s"])
    value = statistics.median(per_step)
    line = {
        "impl": "reference", "metric": "fused logits + top-k rows/s", "value": value,
        "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": case.S_q / value * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (exact e4m3 decode) -> i32", "data": "synthetic",
        "config": {"workload": args.workload, "S_q": case.S_q, "S_kv": case.S_kv, "H": case.H,
                   "D": case.D, "topk": topk},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": info["cores"], "kind": "oracle",
                         "sample": f"{info['rows']} of {case.S_q} rows per step, extrapolated to "
                                   f"the full workload ({info['wall_s']:.1f} s)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_topk(args):
    from fp8_mqa_indexer_gb300 import workloads as wl
    case = wl.topk_config(args.workload)
    for _ in range(args.warmup):
        topk_oracle_sample(case, budget_s=0.3)
    budget = args.ref_budget or max(1.0, min(6.0, 90.0 / max(1, args.steps)))
    per_step, info = [], None
    for _ in range(args.steps):
        info = topk_oracle_sample(case, budget_s=budget)
        per_step.append(info["rows_per_s"])
    value = statistics.median(per_step)
    line = {
        "impl": "reference", "metric": "top-k key selection rows/s", "value": value,
        "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": case.rows / value * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 -> i32", "data": "synthetic",
        "config": {"workload": args.workload, "rows": case.rows, "n_cols": case.n_cols,
                   "topk": case.topk},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": info["cores"], "kind": "oracle",
                         "sample": f"{info['rows']} of {case.rows} rows per step, extrapolated to "
                                   f"the full workload ({info['wall_s']:.1f} s)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def case_bytes(case) -> int:
    """Algorithmic bytes of a dense call: output, q, kv, scales, weights and
    ranges, each once."""
    return (case.S_q * case.ldo * 4 + case.q.numel() + case.kv.numel() + case.kv_scale.numel() * 4
            + case.weights.numel() * 4 + case.S_q * 8)


def e2e_dense_pipelined(args, mqa, torch, dev, case, out, n_chunks: int = 8):
    """Per step: copy the inputs from pinned host memory, compute, copy the
    logits back, with the rows cut into chunks so that the two copy directions
    and the kernel overlap.  Returns (ms per step, h2d bytes, d2h bytes, chunks)."""
    host = {k: v.pin_memory() for k, v in dict(q=case.q, kv=case.kv, s=case.kv_scale, w=case.weights,
                                                ks=case.k_start, ke=case.k_end).items()}
    host_out = torch.empty((case.S_q, case.ldo), dtype=torch.float32, pin_memory=True)
    dv = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    tok = max(1, 256 // case.H)
    per = -(-case.S_q // n_chunks)
    per = -(-per // tok) * tok
    bounds = [(a, min(case.S_q, a + per)) for a in range(0, case.S_q, per)]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def step():
        start = torch.cuda.Event()
        start.record(comp)
        s_in.wait_event(start)
        s_out.wait_event(start)
        with torch.cuda.stream(s_in):
            for k in ("kv", "s"):
                dv[k].copy_(host[k], non_blocking=True)
            ev_in = []
            for a, b in bounds:
                for k in ("q", "w", "ks", "ke"):
                    dv[k][a:b].copy_(host[k][a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in)
                ev_in.append(e)
        ev_out = []
        for (a, b), e in zip(bounds, ev_in):
            comp.wait_event(e)
            mqa.mqa_logits(dv["q"][a:b], dv["kv"], dv["s"], dv["w"][a:b], dv["ks"][a:b],
                           dv["ke"][a:b], out[a:b], clean=case.clean, compressed=case.compressed,
                           ldo=case.ldo, stream=comp)
            e2 = torch.cuda.Event()
            e2.record(comp)
            ev_out.append(e2)
        with torch.cuda.stream(s_out):
            for (a, b), e in zip(bounds, ev_out):
                s_out.wait_event(e)
                host_out[a:b].copy_(out[a:b], non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_out)
        comp.wait_event(done)

    step()
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(comp)
    for _ in range(args.e2e_steps):
        step()
    eb.record(comp)
    torch.cuda.synchronize()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    return ea.elapsed_time(eb) / args.e2e_steps, h2d, host_out.numel() * 4, len(bounds)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dense_2k_32k_h64_d128")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time")
    ap.add_argument("--ref-budget", type=float, default=None,
                    help="oracle seconds per reference step (default: about 90 s in all)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph timing (5 calls per graph, 40 replays)")
    ap.add_argument("--no-fp8-peak", action="store_true",
                    help="skip the live cuBLAS FP8 peak measurement (use bf16 x 2)")
    args = ap.parse_args()
    rank, world, local = dist_env()

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import fp8_mqa_indexer_gb300 as mqa
    from fp8_mqa_indexer_gb300 import build as mqa_build

    assert torch.cuda.is_available(), "bench.py needs a GPU"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    if rank == 0 or world == 1:
        mqa_build.build()
    if pg:
        pg.barrier()
    mqa.load_library()
    if is_fused(args.workload):
        if world > 1:
            raise SystemExit("the fused workloads are measured on one GPU")
        return bench_fused(args, mqa, torch, dev, torch.cuda.current_stream())
    if is_topk(args.workload):
        if world > 1:
            raise SystemExit("the top-k workload is measured on one GPU")
        return bench_topk(args, mqa, torch, dev, torch.cuda.current_stream())
    if is_paged(args.workload):
        if world > 1:
            raise SystemExit("the paged workload is measured on one GPU")
        return bench_paged(args, mqa, torch, dev, torch.cuda.current_stream())
    if is_mx(args.workload):
        if world > 1:
            raise SystemExit("the MX workloads are measured on one GPU")
        return bench_mx(args, mqa, torch, dev, torch.cuda.current_stream())

    case = make_case(args.workload)
    valid = int(case.valid_counts().sum())
    flops = valid * 2.0 * case.H * case.D
    q, kv = case.q.to(dev), case.kv.to(dev)
    s, w = case.kv_scale.to(dev), case.weights.to(dev)
    ks, ke = case.k_start.to(dev), case.k_end.to(dev)
    out = torch.empty((case.S_q, case.ldo), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        mqa.mqa_logits(q, kv, s, w, ks, ke, out, clean=case.clean, compressed=case.compressed,
                       ldo=case.ldo)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert mqa.device_status() == 0

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[local].strip() if vis else str(local))
    sampler.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        pre_spin(torch)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    times_ms = [a.elapsed_time(b) for a, b in ev]
    assert mqa.device_status() == 0
    total_ms = sum(times_ms)
    if pg:
        t = torch.tensor([total_ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / args.steps
    value = flops * world / (ms_per_step * 1e-3) / 1e12

    # End to end through the public call, from pinned host buffers: the rows
    # are cut into chunks whose host->device copies, mqa_logits calls and
    # device->host copies of the logits run on three streams, so that copies in
    # both directions overlap the kernel (the keys and their scales go first;
    # every chunk's call needs them).
    e2e_ms, h2d, d2h, n_chunks = e2e_dense_pipelined(args, mqa, torch, dev, case, out)
    e2e_value = flops * world / (e2e_ms * 1e-3) / 1e12

    graph = None
    if not args.no_graph:
        graph = graph_timing(torch, lambda o: mqa.mqa_logits(q, kv, s, w, ks, ke, o, clean=case.clean,
                                                             compressed=case.compressed,
                                                             ldo=case.ldo), out)
        graph["tflops_at_median"] = flops / (graph["median_ms"] * 1e-3) / 1e12
    assert mqa.device_status() == 0

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0

    peaks, peaks_src = load_peaks()
    nominal_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    fp8 = None if args.no_fp8_peak else measure_fp8_peak(torch, dev)
    peak, peak_source = fp8_roofline_peak(fp8, nominal_peak, peaks_src)
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    traffic = recorded_traffic(args.workload)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    at_clock = (FP8_FLOP_PER_SM_CLK * n_sm * clocks["sm_mhz"] * 1e6 / 1e12
                if clocks.get("sm_mhz") else None)
    line = {
        "metric": "MQA logits TFLOP/s (valid logits x 2*H*D)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "S_q": case.S_q, "S_kv": case.S_kv, "H": case.H,
                   "D": case.D, "valid_logits": valid, "clean": case.clean,
                   "compressed": case.compressed, "ldo": case.ldo,
                   "l2": "flushed (256 MiB write) before every timed step",
                   "parallelism": f"replicas x{world} (independent rows, no collective)"},
        "valid_logits_per_s": valid * world / (ms_per_step * 1e-3),
        **percentiles(times_ms),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes": case_bytes(case),
                     "peak_source": peak_source,
                     "peak_bf16x2": nominal_peak, "frac_bf16x2": achieved / nominal_peak,
                     "peak_at_kernel_clock": at_clock,
                     "frac_at_kernel_clock": achieved / at_clock if at_clock else None,
                     "at_clock_basis": f"{FP8_FLOP_PER_SM_CLK} FLOP per SM per cycle x {n_sm} SMs x "
                                       "median SM clock of the timed region"},
        "fp8_peak": fp8,
        "graph_timing": graph,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": f"pinned host buffers, {n_chunks} row chunks, copies in both directions "
                       "overlapping the calls on three streams"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        info = oracle_sample(case, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": info["tflops"], "unit": "TFLOP/s", "cores": info["cores"],
                                "kind": "oracle",
                                "sample": f"{info['rows']} of {case.S_q} rows ({info['wall_s']:.1f} s"
                                          f" of oracle time), throughput extrapolated"}
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
