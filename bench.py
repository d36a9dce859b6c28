#!/usr/bin/env python3
"""Benchmark of the replica-integrity scan (weight fingerprint check) on GB300.

Metric: fingerprint-scan GB/s (and % of HBM peak, ms per pass) on the
~1.04e9-parameter layout (24 layers, d=1792, ffn=7168, vocab=32000, untied
embedding and head), float32 weights, 3 replicas resident in HBM.

One step = one data-parallel weight check: every rank fingerprints its 3
local copies (sdc_fingerprint: the persistent scan kernel plus its combine),
the [3, 195, 2] tables are all-gathered (no exchange with one rank), and
sdc_vote runs on the gathered table on every rank.  Algorithmic bytes per step = every weight byte of every
replica read once = 12,475,438,080 bytes; inputs are ~97x the 129 MB L2, so
no flush is needed between steps.  The other hot-path rows (fused gradient
average-scan on 4 bf16 buffers of the same layout, xorsum with pair compare)
are timed in the same run and reported under "rows".

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 it is launched with torch.distributed.run, one rank per GPU; every
rank holds 3 copies of the same weights (weak scaling: the work per GPU is
fixed), rank 0's copies hold the one flipped bit, the tables are all-gathered
with NCCL and every rank votes over all 3N copies; rank 0 prints one JSON
line with the whole-job throughput.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fingerprint-scan GB/s and % of GB300 HBM peak; ms/pass at ~1B params"
WORKLOAD = "1b_fp32_3replicas"


# ---------------------------------------------------------------- distributed helpers
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """MAX of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(bytes_per_step_per_rank: int, world: int, ms_per_step_max: float) -> float:
    """GB/s of the whole job: every rank's bytes over the slowest rank's time."""
    return bytes_per_step_per_rank * world / (ms_per_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "active": parts[4],
                             "hw": parts[5], "hwt": parts[6], "swt": parts[7], "pcap": parts[8]})
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                            ("pcap", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def scan_traffic(layers: int):
    """DRAM bytes per launch of the scan kernel from the committed ncu summary,
    scaled to this workload, or None when the kernel source changed since."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "fp_scan_traffic.json")
    src = os.path.join(ROOT, "silent_corruption_checksums_gb300", "csrc", "sdc_fp.cu")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("source_sha256") != hashlib.sha256(open(src, "rb").read()).hexdigest():
        return None
    return d["dram_bytes_per_launch"] * d.get("scale_to_full", 1.0) if layers == 24 else None


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", 1900.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ---------------------------------------------------------------- CPU baseline (the oracle)
def cpu_info() -> dict:
    """Host cores and CPU model (lscpu's model name, else the platform's processor string)."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"nproc": os.cpu_count() or 1, "model": model or platform.processor() or platform.machine()}


def host_bits(t):
    """A device tensor's raw bits as a host numpy array (uint16 for 2-byte, uint32 for 4-byte elements)."""
    import numpy as np
    import torch
    t = t.contiguous()
    if t.element_size() == 2:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.element_size() == 4:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.cpu().numpy()


def oracle_rate(work, nbytes: int, sample: str, unit: str = "GB/s", single=None, single_bytes: int = 0,
                single_sample: str = "") -> dict:
    """Time the oracle on all host cores (work(threads)) and single-threaded (single(1), a smaller sample)."""
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    work(threads)
    dt = time.perf_counter() - t0
    out = {"value": nbytes / dt / (1e9 if unit == "GB/s" else 1e12), "unit": unit, "cores": threads,
           "kind": "oracle", "seconds": dt, "sample": sample, "cpu": cpu_info()}
    if single is not None:
        t0 = time.perf_counter()
        single(1)
        ds = time.perf_counter() - t0
        out["single_thread"] = {"value": single_bytes / ds / (1e9 if unit == "GB/s" else 1e12), "unit": unit,
                                "cores": 1, "seconds": ds, "sample": single_sample}
    return out


def oracle_stream_rate(tensors, fn, limit_bytes: int, single_limit: int, what: str) -> dict:
    """The oracle over device tensors streamed to the host one at a time (the copies are not
    timed): fn(host_bits, threads) on all cores for the first ~limit_bytes, and on one core
    for the first ~single_limit bytes."""
    threads = os.cpu_count() or 1
    t_all = t_one = 0.0
    nb_all = nb_one = n_all = n_one = 0
    for t in tensors:
        if nb_all >= limit_bytes:
            break
        h = host_bits(t)
        t0 = time.perf_counter()
        fn(h, threads)
        t_all += time.perf_counter() - t0
        nb_all += h.nbytes
        n_all += 1
        if nb_one < single_limit:
            t0 = time.perf_counter()
            fn(h, 1)
            t_one += time.perf_counter() - t0
            nb_one += h.nbytes
            n_one += 1
    return {"value": nb_all / t_all / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle", "seconds": t_all,
            "sample": f"{what}: the first {n_all} tensors ({nb_all} bytes), each copied to the host before "
                      "its timed compute", "cpu": cpu_info(),
            "single_thread": {"value": nb_one / t_one / 1e9, "unit": "GB/s", "cores": 1, "seconds": t_one,
                              "sample": f"the first {n_one} tensors ({nb_one} bytes)"}}


def cpu_baseline_sample(host_tensors, threads: int) -> dict:
    """Time the oracle's fingerprint over host copies of a sample of the workload."""
    import oracle
    import numpy as np
    arrays = [t.numpy().view(np.uint32) if t.dtype.itemsize == 4 else t.numpy() for t in host_tensors]
    nbytes = sum(a.nbytes for a in arrays)
    t0 = time.perf_counter()
    for a in arrays:
        oracle.fingerprint(a, threads=threads)
    dt = time.perf_counter() - t0
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seconds": dt, "bytes": nbytes}


def run_reference(args) -> None:
    """The reference arm: the CPU oracle on the whole step of the same workload (3 float32
    copies of the 1b layout, 12.5 GB per step) on all host cores."""
    rank, world, local = dist_env()
    if world > 1 and rank != 0:
        return
    import numpy as np
    import torch
    import sdc_workloads as W
    import oracle
    threads = os.cpu_count() or 1
    oracle.build()
    # the workload, made on the GPU when there is one (faster), then held in host memory
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    layout = W.layout_1b(args.layers)
    copies = []
    for r in range(3):
        g = W.generator(1 + r, dev)
        copies.append([W.normal(shape, 0.02, torch.float32, g, dev).cpu().numpy().view(np.uint32)
                       for _, shape in layout])
        if dev.type == "cuda":
            torch.cuda.empty_cache()
    nbytes = sum(a.nbytes for c in copies for a in c)

    def step():
        for c in copies:
            for a in c:
                oracle.fingerprint(a, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    sample = f"the whole step: 3 copies x {len(layout)} tensors, {nbytes} bytes of float32 weights"
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int64", "data": "synthetic",
            "config": {"workload": WORKLOAD if args.layers == 24 else f"{WORKLOAD}_{args.layers}layers",
                       "sample": sample},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample, "cpu": cpu_info()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def run_only_row(args) -> None:
    """Time one row alone (profiling helper): prints a small JSON line."""
    import numpy as np
    import torch
    import sdc_workloads as W
    import silent_corruption_checksums_gb300 as sdc
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rows = bench_rows(args, dev, torch.cuda.current_stream(), measured_peaks(), sdc, W, torch, np,
                      only=args.only)
    print(json.dumps({"only": args.only, "layers": args.layers, "rows": rows}), flush=True)


def run_ours(args) -> None:
    import numpy as np
    import torch
    import sdc_workloads as W
    import silent_corruption_checksums_gb300 as sdc
    from silent_corruption_checksums_gb300 import dp

    if args.only:
        return run_only_row(args)
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks = measured_peaks()
    stream = torch.cuda.current_stream()

    # ---- workload: every rank holds the same 3 float32 copies of the 1b layout (data parallelism keeps
    # the copies bit-identical); one seeded bit flip in one copy, on rank 0 only
    w = W.weights_1b(dev, seed=1, n_layers=args.layers)
    reps, truth = w["replicas"], w["truth"]
    if rank != 0:  # this rank's copies are all clean
        W.xor_element(reps[truth["replica"]][truth["tensor"]], truth["element"], 1 << truth["bit"])
    R, T = len(reps), len(reps[0])
    bytes_per_step = sum(t.numel() * t.element_size() for ts in reps for t in ts)
    # the data-parallel weight check: fingerprint the local copies, all-gather the [T, 2] tables (none
    # with one rank), the same strict-majority vote on every rank
    wc = dp.WeightCheck(reps, chunk_bytes=args.chunk_bytes)
    plan = wc.plan

    def step():
        wc.fingerprint(stream)
        wc.gather_and_vote(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    # correctness of what is timed: every rank names rank 0 and the flipped copy
    res = wc.result()
    ok = res == {"diverged": True, "suspects": [0], "suspect_replicas": [truth["replica"]]}

    # ---- timed region: K steps, events around each fingerprint call
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            wc.fingerprint(stream)
            ev[i][1].record(stream)
            wc.gather_and_vote(stream)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = start.elapsed_time(stop)
    ms_step = max_over_ranks(elapsed_ms / args.steps, world, dev)
    fp_times = [a.elapsed_time(b) for a, b in ev]
    fp_ms = statistics.median(fp_times)
    clocks = clk.summary()
    value = whole_job_rate(bytes_per_step, world, ms_step)
    achieved = bytes_per_step / (fp_ms * 1e-3) / 1e9
    launches_per_step = (2 if plan.n_chunks else 1) + 1  # scan + combine, vote (+ a memset node)

    rows = {}
    e2e = None
    cpu = None
    if not args.quick:
        e2e_set = E2E(args, reps, dp, torch)
        if world == 1:  # the other rows are single-GPU workloads, measured once
            rows = bench_rows(args, dev, stream, peaks, sdc, W, torch, np)
        e2e = e2e_set.run(args, wc.table, stream, torch, bytes_per_step, world, dev)
        e2e_set.close(torch)
        if rank == 0 and world == 1:
            cpu = bench_cpu(reps, torch)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "int64", "data": "synthetic",
                "config": {"workload": WORKLOAD if args.layers == 24 else f"{WORKLOAD}_{args.layers}layers",
                           "params_per_replica": W.layout_numel(w["layout"]),
                           "replicas": R, "tensors": T, "weights": "float32 N(0,0.02), one seeded bit flip",
                           "parallelism": f"data-parallel weight check: {world} rank(s) x {R} local copies, "
                                          "all-gather of the [T, 2] tables, the same vote on every rank",
                           "copies_voted": world * R,
                           "bytes_per_step": bytes_per_step, "chunk_bytes": plan_chunk_bytes(args),
                           "grid": plan.grid, "block": plan.block, "n_chunks": plan.n_chunks,
                           "l2": "inputs 12.5 GB per step >> 129 MB L2; no flush between steps",
                           "vote_names_flipped_replica": ok},
                "pct_hbm_peak": 100.0 * value / world / peaks["hbm_gbs"],
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": achieved / peaks["hbm_gbs"],
                             "traffic": args.traffic if args.traffic is not None else scan_traffic(args.layers),
                             "kernel": "fp_scan_kernel (+ fp_combine_kernel, timed together as sdc_fingerprint)",
                             "timing": f"median of {args.steps} per-call CUDA-event durations",
                             "mean_ms": statistics.mean(fp_times), "median_ms": fp_ms,
                             "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"},
                "kernel_ms": fp_ms, "gpu_launches": launches_per_step * args.steps,
                "clocks": clocks, "rows": rows, "e2e": e2e, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    wc.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def plan_chunk_bytes(args) -> int:
    return args.chunk_bytes or 16384


def _time_loop(fn, steps, stream, torch):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def _graph_of(fn, torch):
    """fn's launches captured once in a CUDA graph (fn launches on the current stream; warmed up on a
    side stream first, as capture requires)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _time_calls_evicted(fn, steps, stream, torch):
    """Median CUDA-event time of fn, each call timed alone after a read pass over a 512 MiB buffer
    that is not one of its inputs: whatever the call left in the 126 MiB L2 is evicted, and no dirty
    lines are left for the call to write back."""
    evict = torch.ones(512 << 20, dtype=torch.uint8, device=stream.device)
    sink = torch.zeros((), dtype=torch.int64, device=stream.device)
    for _ in range(3):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            sink.copy_(evict.view(torch.int64).sum())
            a.record(stream)
            fn()
            b.record(stream)
    torch.cuda.synchronize()
    del evict
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def bench_rows(args, dev, stream, peaks, sdc, W, torch, np, only=None) -> dict:
    """The other rows of the hot path, each timed on its own workload."""
    rows = {}
    if only in ("fingerprint_8b", "fingerprint_stress", "xorsum_pairs"):
        return bench_big_rows(args, dev, stream, peaks, sdc, W, torch, only)
    if only == "abft_gemm":
        return bench_abft_row(args, dev, stream, peaks, sdc, W, torch)
    if only == "abft_wgrad":
        return bench_wgrad_row(args, dev, stream, peaks, sdc, W, torch)
    if only == "attn_invariant":
        return bench_attn_row(args, dev, stream, peaks, sdc, W, torch)
    import oracle
    oracle.build()
    # fused gradient average-scan on 4 bf16 buffers of the 1b layout
    g = W.grads_flat(W.layout_numel(W.layout_1b(args.layers)), 4, torch.bfloat16, 1e-3, dev, seed=3)
    bufs = g["bufs"]
    n = bufs[0].numel()
    out = torch.empty_like(bufs[0])
    need = sdc.sdc_grad_average_scan_workspace_size(n, 4, sdc.DTYPE_BF16)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

    def avg_step():
        sdc.grad_average_scan(bufs, out=out, stream=stream, ws=ws)

    ms = _time_loop(avg_step, max(5, args.steps // 10), stream, torch) if only in (None, "grad_average_scan") \
        else None
    nbytes = 5 * n * 2
    # the oracle's samples: the first elements of every buffer (all cores), a quarter of that (one core)
    ns = min(n, 1 << 26)
    hb = [host_bits(b[:ns]) for b in bufs]

    def oracle_avg(k):
        def run(threads):
            avg = oracle.average([h[:k] for h in hb], "bf16", threads=threads)
            for h in hb:
                oracle.grad_stats(h[:k], "bf16", threads=threads)
            oracle.grad_stats(avg, "bf16", threads=threads)
        return run

    if ms is not None:
        rows["grad_average_scan"] = {"workload": "4 x bf16 local grads of the 1b layout (N(0,1e-3), rate-1e-7 "
                                     "NaN/Inf/2^70 in buffer 2)", "ms": ms, "bytes": nbytes,
                                     "GB_s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"],
                                     "cpu_baseline": oracle_rate(
                                         oracle_avg(ns), 5 * ns * 2,
                                         f"average + 5 scans of the first {ns} elements of each buffer",
                                         single=oracle_avg(ns // 4), single_bytes=5 * (ns // 4) * 2,
                                         single_sample=f"the first {ns // 4} elements")}
    # the same buffers as one plan: pre-average scan only
    if only in (None, "grad_scan"):
        gplan = sdc.Plan([[b] for b in bufs])
        stats = torch.empty((4, sdc.GRAD_STATS_DTYPE.itemsize), dtype=torch.uint8, device=dev)
        ms = _time_loop(lambda: gplan.grad_scan(out=stats, stream=stream), max(5, args.steps // 10), stream,
                        torch)
        nbytes = 4 * n * 2

        def oracle_scan(k):
            return lambda threads: [oracle.grad_stats(h[:k], "bf16", threads=threads) for h in hb]

        rows["grad_scan"] = {"workload": "4 x bf16 local grads of the 1b layout", "ms": ms, "bytes": nbytes,
                             "GB_s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"],
                             "cpu_baseline": oracle_rate(
                                 oracle_scan(ns), 4 * ns * 2, f"scans of the first {ns} elements of each buffer",
                                 single=oracle_scan(ns // 4), single_bytes=4 * (ns // 4) * 2,
                                 single_sample=f"the first {ns // 4} elements")}
        del gplan
    if only in (None, "adamw_fingerprint"):
        rows.update(bench_adamw_row(args, dev, stream, peaks, sdc, W, torch))
    if only in (None, "xorsum"):
        # xorsum + pair compare of 4 bf16 buffers against copies (original vs recomputed)
        rec = [b.clone() for b in bufs]
        W.xor_element(rec[1], 12345, 1 << 3)
        xplan = sdc.Plan([list(bufs), rec])
        xo = torch.empty((2, 4), dtype=torch.int64, device=dev)

        def xor_step():
            xplan.xorsum(out=xo, stream=stream)
            sdc.xorsum_compare(xo[0], xo[1], stream=stream)

        ms = _time_loop(xor_step, max(5, args.steps // 10), stream, torch)
        nbytes = 8 * n * 2
        hr = host_bits(rec[1][:ns])

        def oracle_xor(k):
            def run(threads):
                xa = [oracle.xorsum(h[:k], threads=threads) for h in hb]
                xb = [oracle.xorsum(h[:k], threads=threads) for h in (hb[0], hr, hb[2], hb[3])]
                oracle.xorsum_compare(xa, xb)
            return run

        rows["xorsum"] = {"workload": "xorsum of 4 bf16 grad buffers and their recomputed copies + compare",
                          "ms": ms, "bytes": nbytes, "GB_s": nbytes / ms / 1e6,
                          "frac_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"],
                          "cpu_baseline": oracle_rate(
                              oracle_xor(ns), 8 * ns * 2, f"the first {ns} elements of the 4 buffers and 4 copies",
                              single=oracle_xor(ns // 4), single_bytes=8 * (ns // 4) * 2,
                              single_sample=f"the first {ns // 4} elements")}
        del xplan, rec
    del g, bufs, out, ws, hb
    torch.cuda.empty_cache()
    if only in (None, "abft_gemm"):
        rows.update(bench_abft_row(args, dev, stream, peaks, sdc, W, torch))
    if only in (None, "abft_wgrad"):
        rows.update(bench_wgrad_row(args, dev, stream, peaks, sdc, W, torch))
    if only in (None, "attn_invariant"):
        rows.update(bench_attn_row(args, dev, stream, peaks, sdc, W, torch))
    if not getattr(args, "no_big_rows", False):
        rows.update(bench_big_rows(args, dev, stream, peaks, sdc, W, torch, only))
    return rows


def bench_adamw_row(args, dev, stream, peaks, sdc, W, torch) -> dict:
    """Fused clip + AdamW step + fingerprint on one fp32 replica of the 1b layout, bf16 averaged gradient."""
    layout = W.layout_1b(args.layers)
    gen = W.generator(21, dev)
    weights = [[W.normal(s, 0.02, torch.float32, gen, dev) for _, s in layout]]
    grads = [W.normal(s, 1e-3, torch.bfloat16, gen, dev) for _, s in layout]
    m = [[torch.zeros(s, dtype=torch.float32, device=dev) for _, s in layout]]
    v = [[torch.zeros(s, dtype=torch.float32, device=dev) for _, s in layout]]
    plan = sdc.Plan(weights)
    opt = sdc.AdamWFingerprint(plan, grads, m, v)
    fp = torch.empty((1, len(layout), 2), dtype=torch.int64, device=dev)
    hp = {"lr": 3e-4, "beta1": 0.9, "beta2": 0.95, "eps": 1e-8, "weight_decay": 0.1, "max_grad_norm": 1.0,
          "step": 1, "clip": 0}
    ms = _time_loop(lambda: opt.step(hp, out=fp, stream=stream), max(5, args.steps // 20), stream, torch)
    ms_fp = _time_loop(lambda: plan.fingerprint(out=fp, stream=stream), max(5, args.steps // 20), stream, torch)
    n = W.layout_numel(layout)
    nbytes = n * (4 + 2 + 4 + 4 + 4 + 4 + 4)  # read p, g(bf16), m, v; write p, m, v
    out = {"adamw_fingerprint": {"workload": "1 fp32 replica of the 1b layout, bf16 averaged gradient, fp32 moments: "
                                 "AdamW step + fingerprint of the written weights in one pass",
                                 "ms": ms, "bytes": nbytes, "GB_s": nbytes / ms / 1e6,
                                 "frac_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"],
                                 "separate_fingerprint_reread_ms": ms_fp}}
    # the oracle (one core: it is plain scalar C) on the first 2^24 elements of the first tensor
    import numpy as np
    import oracle
    k = min(1 << 24, weights[0][0].numel())
    p_h = host_bits(weights[0][0]).reshape(-1)[:k].view(np.float32).copy()
    g_h = host_bits(grads[0]).reshape(-1)[:k].copy()
    m_h, v_h = np.zeros(k, dtype=np.float32), np.zeros(k, dtype=np.float32)
    t0 = time.perf_counter()
    oracle.adamw_step(p_h, g_h, "bf16", m_h, v_h, hp, None)
    dt = time.perf_counter() - t0
    out["adamw_fingerprint"]["cpu_baseline"] = {
        "value": k * 26 / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle", "seconds": dt,
        "sample": f"the AdamW update of the first {k} elements of the first tensor (the oracle is single-threaded)",
        "cpu": cpu_info()}
    opt.close()
    del plan, weights, grads, m, v
    torch.cuda.empty_cache()
    return out


def bench_abft_row(args, dev, stream, peaks, sdc, W, torch) -> dict:
    """GEMM with the in-kernel accumulator row checksum (the sensor) and its check (the
    verifier) on the 8b layout's MLP up-projection, with cuBLAS's plain GEMM beside it."""
    M, N, K = W.GEMM_8B_UP
    ops = W.gemm_operands(M, N, K, dev, seed=6)
    A, Wt = ops["A"], ops["W"]
    g = sdc.AbftGemm(M, N, K, dev)
    reps = max(10, args.steps // 10)
    ms_gemm = _time_loop(lambda: g.gemm(A, Wt, stream=stream), reps, stream, torch)
    # the verifier reads 185 MB: each call timed alone with the L2 emptied of its inputs before it (and
    # back to back beside it)
    ms_verify = _time_calls_evicted(lambda: g.verify(A, Wt, stream=stream), reps, stream, torch)
    ms_verify_b2b = _time_loop(lambda: g.verify(A, Wt, stream=stream), reps, stream, torch)
    gc = sdc.AbftGemm(M, N, K, dev, columns=True)  # the row + column configuration
    ms_gemm_rc = _time_loop(lambda: gc.gemm(A, Wt, stream=stream), reps, stream, torch)
    ms_verify_rc = _time_calls_evicted(lambda: gc.verify(A, Wt, stream=stream), reps, stream, torch)
    ms_cublas = _time_loop(lambda: torch.matmul(A, Wt.t()), reps, stream, torch)
    # the row check fused into the GEMM: W's column sums once per weight version, then the GEMM whose
    # extra warps form the reference beside the product
    # (the plain and the fused GEMM in alternating rounds, so that both see the same power state)
    ms_wsums = _time_loop(lambda: g.weight_sums(Wt, stream=stream), reps, stream, torch)
    pairs = [(_time_loop(lambda: g.gemm(A, Wt, stream=stream), reps, stream, torch),
              _time_loop(lambda: g.gemm_checked(A, Wt, stream=stream), reps, stream, torch)) for _ in range(3)]
    ms_plain_alt = statistics.median(p[0] for p in pairs)
    ms_fused = statistics.median(p[1] for p in pairs)
    torch.cuda.synchronize()
    fused_flagged = int(g.summary[0])
    g.gemm(A, Wt, stream=stream)
    g.verify(A, Wt, stream=stream)
    torch.cuda.synchronize()
    flops = 2.0 * M * N * K
    tf = flops / (ms_gemm * 1e-3) / 1e12
    vbytes = (M + N) * K * 2
    out = {"abft_gemm": {"workload": f"C = A W^T, bf16, M={M} tokens x N={N} x K={K} (8b MLP up-projection), "
                         "A N(0,1), W N(0,0.02); row checksum from the fp32 accumulator + check vs A(W^T 1)",
                         "gemm_ms": ms_gemm, "tflops": tf, "frac_bf16_peak": tf / peaks["bf16_tflops"],
                         "peak_tflops": peaks["bf16_tflops"],
                         "peak_kind": f"burst bf16 (MEASURED_PEAKS.json bf16_tflops, {peaks['source']})",
                         "verify_ms": ms_verify, "verify_GB_s": vbytes / ms_verify / 1e6,
                         "verify_frac_hbm": vbytes / ms_verify / 1e6 / peaks["hbm_gbs"],
                         "verify_timing": "each call alone after a 512 MiB read pass (its inputs out of L2), median",
                         "verify_back_to_back_ms": ms_verify_b2b,
                         "row_col_gemm_ms": ms_gemm_rc, "row_col_tflops": flops / (ms_gemm_rc * 1e-3) / 1e12,
                         "row_col_over_row_only": ms_gemm_rc / ms_gemm - 1.0, "row_col_verify_ms": ms_verify_rc,
                         "row_col_clean_flagged": [int(gc.summary[0]), int(gc.summary[1])],
                         "cublas_plain_gemm_ms": ms_cublas,
                         "cublas_tflops": flops / (ms_cublas * 1e-3) / 1e12,
                         "fused_row_check_gemm_ms": ms_fused, "fused_over_gemm": ms_fused / ms_plain_alt - 1.0,
                         "fused_vs_plain_rounds_ms": [[round(a, 4), round(b, 4)] for a, b in pairs],
                         "separate_row_check_over_gemm": ms_verify / ms_gemm,
                         "weight_sums_ms": ms_wsums, "fused_clean_rows_flagged": fused_flagged,
                         "clean_rows_flagged": int(g.summary[0]), "aborted": int(g.aborted[0]),
                         "max_residual_over_bound": float((g.residual.abs() / g.bound).max())}}
    # the oracle (float64, numpy's BLAS on all host cores) on the first 64 rows of A
    import oracle
    ms_rows = 64
    A_h = host_bits(A[:ms_rows]).reshape(ms_rows, K)
    W_h = host_bits(Wt).reshape(N, K)
    t0 = time.perf_counter()
    C_ref = oracle.abft_product(A_h, W_h)
    oracle.abft_verify(oracle.abft_row_checksum(C_ref), A_h, W_h)
    dt = time.perf_counter() - t0
    out["abft_gemm"]["cpu_baseline"] = {
        "value": 2.0 * ms_rows * N * K / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count() or 1,
        "kind": "oracle", "seconds": dt, "cpu": cpu_info(),
        "sample": f"the product, row checksums and check of the first {ms_rows} rows of A (float64; the "
                  "matrix product runs on numpy's BLAS with its default threads)"}
    del g, gc, ops, A, Wt, A_h, W_h, C_ref
    torch.cuda.empty_cache()
    return out


def bench_wgrad_row(args, dev, stream, peaks, sdc, W, torch) -> dict:
    """The weight-gradient form of the GEMM checksum, dW = dY^T X from token-major operands, with
    row and column checksums (the configuration that covers wgrad) and their check, on the 8b
    layout's MLP up-projection, with cuBLAS's plain dY^T X beside it."""
    T, N, K = W.GEMM_8B_UP
    ops = W.wgrad_operands(T, N, K, dev, seed=10)
    dY, X = ops["dY"], ops["X"]
    a = sdc.AbftWgrad(T, N, K, dev)
    reps = max(10, args.steps // 10)
    ms_gemm = _time_loop(lambda: a.gemm(dY, X, stream=stream), reps, stream, torch)
    ms_verify = _time_calls_evicted(lambda: a.verify(dY, X, stream=stream), reps, stream, torch)
    ms_verify_b2b = _time_loop(lambda: a.verify(dY, X, stream=stream), reps, stream, torch)
    ms_cublas = _time_loop(lambda: torch.matmul(dY.t(), X), reps, stream, torch)
    torch.cuda.synchronize()
    flops = 2.0 * T * N * K
    tf = flops / (ms_gemm * 1e-3) / 1e12
    vbytes = 2 * (N + K) * T * 2  # each operand read twice: once for its row sums, once for its column sums
    out = {"abft_wgrad": {"workload": f"dW = dY^T X, bf16, T={T} tokens, dY [T, N={N}] N(0, 2^-10), X [T, K={K}] "
                          "N(0,1), token-major (8b MLP up-projection's weight gradient); row + column checksums from "
                          "the fp32 accumulator + check vs dY^T (X 1) and (dY 1)^T X",
                          "gemm_ms": ms_gemm, "tflops": tf, "frac_bf16_peak": tf / peaks["bf16_tflops"],
                          "verify_ms": ms_verify, "verify_GB_s": vbytes / ms_verify / 1e6,
                          "verify_frac_hbm": vbytes / ms_verify / 1e6 / peaks["hbm_gbs"],
                          "verify_timing": "each call alone after a 512 MiB read pass (its inputs out of L2), median",
                          "verify_back_to_back_ms": ms_verify_b2b,
                          "cublas_plain_gemm_ms": ms_cublas, "cublas_tflops": flops / (ms_cublas * 1e-3) / 1e12,
                          "clean_flagged": [int(a.summary[0]), int(a.summary[1])], "aborted": int(a.aborted[0]),
                          "max_residual_over_bound": max(float((a.residual.abs() / a.bound).max()),
                                                         float((a.residual_col.abs() / a.bound_col).max()))}}
    # the oracle on the first 512 tokens: the product and both sides of the check
    import oracle
    ts = 512
    dY_h, X_h = host_bits(dY[:ts]).reshape(ts, N), host_bits(X[:ts]).reshape(ts, K)
    t0 = time.perf_counter()
    dW_ref = oracle.wgrad_product(dY_h, X_h)
    oracle.wgrad_verify(dW_ref.sum(axis=1), dW_ref.sum(axis=0), dY_h, X_h)
    dt = time.perf_counter() - t0
    out["abft_wgrad"]["cpu_baseline"] = {
        "value": 2.0 * ts * N * K / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count() or 1,
        "kind": "oracle", "seconds": dt, "cpu": cpu_info(),
        "sample": f"the product over the first {ts} tokens and both sides of its check (float64; the matrix "
                  "product runs on numpy's BLAS with its default threads)"}
    del a, ops, dY, X, dY_h, X_h, dW_ref
    torch.cuda.empty_cache()
    return out


def bench_attn_row(args, dev, stream, peaks, sdc, W, torch) -> dict:
    """The dV half of the attention backward with the invariant 1^T dV = 1^T dO, on the 8b
    layout's 32 heads of 128 at 4,096 tokens, causal; torch's fused backward (dQ, dK, dV) beside it."""
    BH, L = W.ATTN_8B
    x = W.attn_inputs(BH, L, dev, seed=8, causal=True)
    a = sdc.AttnDvCheck(BH, L, dev)
    reps = max(10, args.steps // 10)
    ms = _time_loop(lambda: a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], True, stream=stream), reps, stream,
                    torch)
    torch.cuda.synchronize()
    flops = 2 * 2.0 * L * L * 128 * BH * 0.5  # S^T = K Q^T and dV = P^T dO over the causal half
    tf = flops / (ms * 1e-3) / 1e12
    q, k, v = (t.unsqueeze(0).clone().requires_grad_(True) for t in (x["Q"], x["K"], x["dO"]))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    g = x["dO"].unsqueeze(0)
    ms_ref = _time_loop(lambda: torch.autograd.grad(o, (q, k, v), g, retain_graph=True), reps, stream, torch)
    out = {"attn_invariant": {"workload": f"{BH} heads x {L} tokens x 128, causal, bf16 Q/K/dO N(0,1), fp32 "
                              "log-sum-exp: dV = P^T dO (P rebuilt from Q K^T and the log-sum-exp) + 1^T dV vs 1^T dO",
                              "ms": ms, "tflops": tf, "frac_bf16_peak": tf / peaks["bf16_tflops"],
                              "peak_tflops": peaks["bf16_tflops"],
                              "clean_columns_flagged": int(a.summary[0]), "aborted": int(a.aborted[0]),
                              "max_residual_over_bound": float((a.residual.abs() / a.bound).max()),
                              "torch_fused_backward_dq_dk_dv_ms": ms_ref}}
    # the oracle (float64, numpy's BLAS on all host cores) on the first head
    import oracle
    Qh, Kh, dOh = (host_bits(x[n][0]).reshape(L, 128) for n in ("Q", "K", "dO"))
    lse_h = x["lse"][0].float().cpu().numpy()
    t0 = time.perf_counter()
    P = oracle.attn_probs(Qh, Kh, lse_h, x["scale"], True)
    oracle.attn_invariant(oracle.attn_dv(P, dOh).sum(axis=0), dOh)
    dt = time.perf_counter() - t0
    out["attn_invariant"]["cpu_baseline"] = {
        "value": flops / BH / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count() or 1, "kind": "oracle",
        "seconds": dt, "cpu": cpu_info(),
        "sample": "the first head: P rebuilt, dV = P^T dO and the invariant (float64, numpy's BLAS with its "
                  "default threads; FLOPs counted as for the GPU row, the causal half)"}
    del a, x, q, k, v, o, P
    torch.cuda.empty_cache()
    # the 8b layout's grouped-query form: its 32 query heads over 8 K/V heads, dV per K/V head
    group = 4
    x = W.attn_inputs(BH, L, dev, seed=9, causal=True, group=group)
    a = sdc.AttnDvCheck(BH, L, dev, group=group)
    ms_g = _time_loop(lambda: a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], True, stream=stream), reps, stream,
                      torch)
    torch.cuda.synchronize()
    tf_g = flops / (ms_g * 1e-3) / 1e12
    out["attn_invariant"].update({"grouped_workload": f"{BH} query heads over {BH // group} K/V heads, the same "
                                                      "shapes and causal mask", "grouped_ms": ms_g,
                                  "grouped_tflops": tf_g, "grouped_frac_bf16_peak": tf_g / peaks["bf16_tflops"],
                                  "grouped_clean_columns_flagged": int(a.summary[0]),
                                  "grouped_aborted": int(a.aborted[0])})
    del a, x
    torch.cuda.empty_cache()
    return out


def bench_big_rows(args, dev, stream, peaks, sdc, W, torch, only) -> dict:
    """Fingerprint rows on the 8b and stress workloads (tens of GB each)."""
    import oracle
    oracle.build()
    rows = {}
    if only in (None, "fingerprint_8b"):
        L8, R8 = getattr(args, "layers_8b", 32), getattr(args, "replicas_8b", 8)
        w8 = W.weights_8b(dev, seed=4, n_replicas=R8, n_layers=L8)
        rows["fingerprint_8b"] = bench_fp_row(
            w8["replicas"], f"8b bf16 layout (T={len(w8['layout'])}, {L8} layers), {R8} replicas, 16-element "
            "perturbation", args, stream, peaks, sdc, torch)
        rows["fingerprint_8b"]["cpu_baseline"] = oracle_stream_rate(
            [t for ts in w8["replicas"] for t in ts], lambda h, th: oracle.fingerprint(h, threads=th), 8 << 30,
            1 << 30, "fingerprint, replica-major")
        del w8
        torch.cuda.empty_cache()
    if only == "xorsum_pairs":  # the pairs alone (profiling): the stress set's pairs, one tensor beside them
        w = W.stress(dev, seed=5, n_tensors=1)
        rows.update(bench_xor_pairs_row(w["pairs"], stream, peaks, sdc, torch, oracle))
        return rows
    if only in (None, "fingerprint_stress"):
        nt = getattr(args, "stress_tensors", 100_000)
        w = W.stress(dev, seed=5, n_tensors=nt)
        rows["fingerprint_stress"] = bench_fp_row(
            w["replicas"], f"{nt:,} tensors (1..1e6 elements, fp32/bf16/fp16, element-aligned packing), 3 replicas",
            args, stream, peaks, sdc, torch)
        rows["fingerprint_stress"]["cpu_baseline"] = oracle_stream_rate(
            [t for ts in w["replicas"] for t in ts], lambda h, th: oracle.fingerprint(h, threads=th), 2 << 30,
            256 << 20, "fingerprint, replica-major")
        rows.update(bench_xor_pairs_row(w["pairs"], stream, peaks, sdc, torch, oracle))
        del w
        torch.cuda.empty_cache()
    return rows


def bench_xor_pairs_row(p, stream, peaks, sdc, torch, oracle) -> dict:
    """Xorsum + compare of the stress set's 1,000 (original, recomputed) pairs."""
    rows = {}
    xplan = sdc.Plan([p["orig"], p["recomp"]])
    xo = torch.empty((2, len(p["orig"])), dtype=torch.int64, device=p["orig"][0].device)

    def xs_step():
        xplan.xorsum(out=xo, stream=stream)
        sdc.xorsum_compare(xo[0], xo[1], stream=stream)

    # the step's four launches (scan, output reset, combine, compare) replayed from a CUDA graph; the same
    # launched on the stream one by one beside it
    gx = _graph_of(lambda: (xplan.xorsum(out=xo), sdc.xorsum_compare(xo[0], xo[1])), torch)
    ms = _time_loop(gx.replay, 20, stream, torch)
    ms_stream = _time_loop(xs_step, 20, stream, torch)
    del gx
    nbytes = sum(t.numel() * t.element_size() for t in p["orig"]) * 2
    ho, hr = [host_bits(t) for t in p["orig"]], [host_bits(t) for t in p["recomp"]]

    def oracle_pairs(threads):
        oracle.xorsum_compare([oracle.xorsum(h, threads=threads) for h in ho],
                              [oracle.xorsum(h, threads=threads) for h in hr])

    rows["xorsum_pairs_stress"] = {"workload": "1,000 (original, recomputed) pairs, sizes 1..1e6, half with a "
                                   "one-bit difference: xorsum + compare", "ms": ms,
                                   "launch": "the step's launches replayed from a CUDA graph",
                                   "stream_launch_ms": ms_stream, "bytes": nbytes,
                                   "GB_s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"],
                                   "cpu_baseline": oracle_rate(oracle_pairs, nbytes, "all 1,000 pairs",
                                                               single=oracle_pairs, single_bytes=nbytes,
                                                               single_sample="all 1,000 pairs")}
    del xplan, ho, hr
    return rows


def bench_fp_row(reps, workload, args, stream, peaks, sdc, torch) -> dict:
    """Fingerprint + vote over a replica set: ms per pass and GB/s of element bytes."""
    plan = sdc.Plan(reps)
    R, T = len(reps), len(reps[0])
    fp = torch.empty((R, T, 2), dtype=torch.int64, device=plan.device)
    vo = (torch.empty(T, dtype=torch.int32, device=plan.device), torch.empty(T, dtype=torch.int64, device=plan.device),
          torch.empty(sdc.VOTE_SUMMARY_DTYPE.itemsize, dtype=torch.uint8, device=plan.device))

    def step():
        plan.fingerprint(out=fp, stream=stream)
        sdc.vote(fp, stream=stream, out=vo)

    ms = _time_loop(step, 20, stream, torch)
    nbytes = sum(t.numel() * t.element_size() for ts in reps for t in ts)
    verdict = sdc.pages_verdict(sdc.decode_summary(vo[2]))
    n_chunks = plan.n_chunks
    del plan
    return {"workload": workload, "ms": ms, "bytes": nbytes, "GB_s": nbytes / ms / 1e6,
            "frac_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"], "n_chunks": n_chunks, "verdict": verdict}


class E2E:
    """The same metric through the public API with the copies in pinned host memory:
    every step copies them to the device, runs the data-parallel weight check
    (fingerprint, all-gather, vote) and reads the table and verdict back.

    Each copy's tensors sit back to back (256-byte aligned) in one host buffer
    allocated pinned and one device buffer; a step moves them in 256 MiB copies.
    The host buffers are written by the CPU, as a caller's host data would be
    (set-up, outside the timed region).  The host link bounds the rate.  The
    check covers views of the device buffers."""

    def __init__(self, args, reps, dp, torch):
        align = 256
        self.offs, total = [], 0
        for t in reps[0]:
            self.offs.append(total)
            total += (t.numel() * t.element_size() + align - 1) // align * align
        self.total, self.n_rep = total, len(reps)
        dev = reps[0][0].device
        self.host, self.dev, views = [], [], []
        for ts in reps:
            h = torch.empty(total, dtype=torch.uint8, pin_memory=True)
            h.zero_()
            d = torch.empty(total, dtype=torch.uint8, device=dev)
            vs = []
            for t, o in zip(ts, self.offs):
                nb = t.numel() * t.element_size()
                v = d[o:o + nb].view(t.dtype).view(t.shape)
                v.copy_(t)
                vs.append(v)
                h[o:o + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())  # CPU writes into the pinned buffer
            h.copy_(h.clone())  # one sequential CPU rewrite of the whole buffer
            self.host.append(h)
            self.dev.append(d)
            views.append(vs)
        self.views = views
        self.wc = dp.WeightCheck(views, chunk_bytes=args.chunk_bytes)

    def run(self, args, table_ref, stream, torch, bytes_per_step, world, dev) -> dict:
        ref = table_ref.cpu()  # the device-resident pass's gathered table: the copied replicas give the same one
        wc = self.wc
        fp_host = torch.empty(wc.table.shape, dtype=wc.table.dtype).pin_memory()
        sum_host = torch.empty(wc.vote_out[2].shape, dtype=torch.uint8).pin_memory()
        sus_host = torch.empty(wc.vote_out[0].shape, dtype=torch.int32).pin_memory()
        piece, total = 256 << 20, self.total

        def e2e_step():
            for h, d in zip(self.host, self.dev):
                for o in range(0, total, piece):
                    e = min(total, o + piece)
                    d[o:e].copy_(h[o:e], non_blocking=True)
            wc.enqueue(stream)
            fp_host.copy_(wc.table, non_blocking=True)
            sus_host.copy_(wc.vote_out[0], non_blocking=True)
            sum_host.copy_(wc.vote_out[2], non_blocking=True)

        # Each step is timed on its own, from its first copy to the host holding the verdict; the
        # host link is shared with the machine's other GPUs, so single steps vary (59 to 220 ms for
        # the same copies on one box) and the median is the rate, the mean and every step beside it.
        steps = max(5, min(12, args.steps // 40))
        e2e_step()
        torch.cuda.synchronize()
        times = []
        for _ in range(steps):
            barrier(world)
            t0 = time.perf_counter()
            e2e_step()
            torch.cuda.synchronize()
            times.append(time.perf_counter() - t0)
        dt = max_over_ranks(statistics.median(times), world, dev)
        same = bool(torch.equal(fp_host, ref))
        d2h = wc.table.numel() * 8 + wc.vote_out[0].numel() * 4 + wc.vote_out[2].numel()
        return {"value": bytes_per_step * world / dt / 1e9, "unit": "GB/s", "ms_per_step": dt * 1e3,
                "statistic": f"median of {steps} steps, each synchronised (max over ranks)",
                "mean_ms": statistics.mean(times) * 1e3, "min_ms": min(times) * 1e3,
                "step_ms": [round(t * 1e3, 2) for t in times],
                "h2d_bytes_per_step": total * self.n_rep, "d2h_bytes_per_step": d2h, "steps": steps,
                "copies_per_step": self.n_rep * ((total + piece - 1) // piece) + 3,
                "per_rank": "h2d and d2h bytes per rank; value = all ranks' bytes over the slowest rank's time",
                "layout": "one pinned buffer per replica, tensors 256-byte aligned, 256 MiB copies",
                "table_matches_device_pass": same}

    def close(self, torch) -> None:
        self.wc.close()
        del self.host, self.dev, self.views
        torch.cuda.empty_cache()


def bench_cpu(reps, torch) -> dict:
    """The oracle on the whole step's bytes (all replicas, all host cores: about 20
    core-seconds), plus a single-threaded figure on the first ~1 GB of replica 0."""
    host = [[t.to("cpu") for t in ts] for ts in reps]
    nbytes = sum(t.numel() * t.element_size() for ts in host for t in ts)
    threads = os.cpu_count() or 1
    r = cpu_baseline_sample([t for ts in host for t in ts], threads)
    r["sample"] = f"the whole step: {len(host)} replicas x {len(host[0])} tensors, {nbytes} bytes"
    r["cpu"] = cpu_info()
    one, nb1 = [], 0
    for t in host[0]:
        one.append(t)
        nb1 += t.numel() * t.element_size()
        if nb1 >= 1 << 30:
            break
    st = cpu_baseline_sample(one, 1)
    r["single_thread"] = {"value": st["value"], "unit": "GB/s", "cores": 1, "seconds": st["seconds"],
                          "sample": f"{len(one)} tensors of replica 0, {nb1} bytes"}
    del host
    return r


def main(argv=None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--chunk-bytes", type=int, default=0)
    ap.add_argument("--quick", action="store_true", help="only the timed fingerprint step (no rows/e2e/cpu)")
    ap.add_argument("--no-big-rows", action="store_true", help="skip the 8b and stress rows")
    ap.add_argument("--only", choices=["grad_average_scan", "grad_scan", "xorsum", "abft_gemm", "abft_wgrad",
                                       "attn_invariant",
                                       "fingerprint_8b", "xorsum_pairs",
                                       "fingerprint_stress", "adamw_fingerprint"], default=None,
                    help="time one row alone (profiling)")
    ap.add_argument("--layers-8b", type=int, default=32,
                    help="decoder layers of the 8b layout (32 = the benchmark workload; fewer for profiling)")
    ap.add_argument("--replicas-8b", type=int, default=8, help="replicas of the 8b row (8; fewer for profiling)")
    ap.add_argument("--stress-tensors", type=int, default=100_000,
                    help="tensors of the stress row (100,000; fewer for profiling)")
    ap.add_argument("--layers", type=int, default=24,
                    help="decoder layers of the 1b layout (24 = the benchmark workload; fewer for profiling)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the scan kernel from an ncu capture, if current")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
