"""Benchmark of the HiSparse swap-in path on GB300.

Metric: top-k resolves/sec (one resolve = one request's K indices for one
layer at one decode step) and miss-row GB/s, against the host->device link
peak measured in the same run.

Default workload: 64 requests, 64K-token contexts, top_k 2048, a 4096-slot hot
buffer per request backed by a 16x pinned host pool, 1152-byte KV rows; the
top-k trace keeps 70 % of each step's indices and draws the rest from
Zipf(1.1).  The 2048-slot buffer of the same trace is measured alongside
(the blog's buffer-size comparison) unless --no-sweep.

One bench step = one call of the whole path (miss detection, LRU victims,
table update, row fetch) for all requests.  The first 10 trace steps (the
empty-buffer start) are run untimed, then --warmup steps untimed, then
--steps timed steps.  L2 is flushed (a 256 MiB write) before every timed step,
outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain sequential implementation the
CUDA path is checked against) on the host cores over the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PRIME_STEPS = 10
# DRAM and host-link bytes of one steady-state launch per (kernel, workload),
# written from ncu captures together with the fingerprint of the kernel's code
# at the time of the capture.  A figure whose fingerprint no longer matches is
# not reported (the kernel has changed since it was measured).
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
# Buffer sizes of the miss-count curve (top-k 2048, so 2048 is the smallest) and its requests.
MISS_CURVE_SLOTS = (2048, 2560, 3072, 4096, 6144, 8192)
MISS_CURVE_REQUESTS = 16
# The files that define each kernel's code.
KERNEL_SOURCES = {
    "hs_resolve_kernel_fused": ["hs_resolve.cu", "hs_internal.h"],
    "hs_resolve_layers_kernel": ["hs_resolve.cu", "hs_internal.h"],
    "hs_copy_kernel": ["hs_copy.cu", "hs_internal.h"],
    "hs_swapin_cluster_kernel": ["hs_resolve.cu", "hs_internal.h"],
}
METRIC = "top-k resolves/sec and miss-row GB/s vs measured H2D peak (1xGB300)"
L2_FLUSH_BYTES = 256 << 20
# Config keys shared word for word by both arms, so that their lines describe
# the same run.
CONFIG_L2 = ("GPU arm: L2 flushed before every timed step (256 MiB write, outside the timed "
             "events); the oracle arm runs on the host cores")
CONFIG_PARALLELISM = "requests sharded over ranks, no collective on the data path"
# The pages' own figures: end-to-end serving results on other hardware, quoted
# as context only (no number of the pages measures the swap-in path itself).
CONTEXT = {
    "note": "the pages' end-to-end serving results on other hardware; context only, not a "
            "kernel result and not the target",
    "figures": [
        {"result": "more than 3x the decode throughput of sparse attention without HiSparse",
         "at": "256 concurrent requests, 32K input / 8K output",
         "hardware": "one node of 8xH200, prefill and decode colocated",
         "settings": "top_k 2048, device_buffer_size 4096, host_to_device_ratio 8",
         "source": "papercache summary, section 1 and section 3; HiSparse blog, introduction "
                   "and 'ベンチマークテスト'"},
        {"result": "up to 5x throughput in long-context settings",
         "at": "a sweep of input / output lengths",
         "hardware": "two nodes of H20, prefill and decode disaggregated",
         "settings": "top_k 2048, device_buffer_size 6144, host_to_device_ratio 10",
         "source": "HiSparse blog, 'ベンチマークテスト'; papercache summary, section 3"},
    ],
}


def _config(wl):
    return {"workload": _workload_desc(wl), "prime_steps_untimed": PRIME_STEPS, "l2": CONFIG_L2,
            "parallelism": CONFIG_PARALLELISM}


def _code_fingerprint(names):
    """First 16 hex digits of the SHA-256 of the given csrc files' code, with
    comments and whitespace removed (a comment edit leaves it unchanged)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "hierarchical_kv_cache_hs_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(name.encode() + b"\0" + " ".join(text.split()).encode() + b"\0")
    return h.hexdigest()[:16]


def dram_traffic(kernel, workload):
    """(DRAM read + write bytes, host-link read bytes, note) of one launch of
    `kernel` on `workload` from the traffic file, or (None, None, why not)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    except OSError:
        return None, None, "no ncu capture on file"
    now = _code_fingerprint(KERNEL_SOURCES[kernel])
    for r in rows:
        if len(r) >= 7 and r[0] == kernel and r[1] == workload:
            if r[5] != now:
                return None, None, ("stale: captured on kernel code %s, the code is now %s"
                                    % (r[5], now))
            return int(r[2]) + int(r[3]), int(r[4]), ("ncu capture of one steady-state launch at "
                                                      "commit %s, kernel code %s" % (r[6], now))
    return None, None, "no ncu capture of this kernel on this workload"


def _workload_desc(wl):
    return ("%s: B=%d requests, ctx %d tokens, top_k %d, buffer %d slots, host pool %dx buffer, "
            "resident tail %d, %d layer(s), row %d B, trace %d%% carry-over / %d%% Zipf(%.1f) / rest %s, "
            "seed %d" % (wl.name, wl.B, wl.C, wl.K, wl.S, wl.host_ratio, wl.T, wl.layers,
                         wl.row_bytes, wl.carry_pct, wl.zipf_pct, wl.zipf_a,
                         ["Zipf", "uniform", "recent window %d" % wl.recent][wl.third], wl.seed))


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the measured region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_path: str = None):
        self.proc = None
        self.lines = []
        self.path = out_path
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if self.path:
            with open(self.path, "w") as f:
                f.write("sm_mhz,max_sm_mhz,power_w,active,hw_slowdown,hw_thermal,sw_thermal,sw_power_cap\n")
                f.write(out)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r[2] > 250.0] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in loaded:
            for n, v in zip(names, r[3][1:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded)}


# ---------------------------------------------------------------- peaks
def measure_h2d_peak(torch, hs, nbytes=1 << 30, reps=5):
    """Best of `reps` for a pinned->device cudaMemcpyAsync and for the zero-copy read kernel."""
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    host.fill_(3)
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best_ce = best_zc = float("inf")
    for _ in range(reps):
        torch.cuda.synchronize()
        e0.record()
        dev.copy_(host, non_blocking=True)
        e1.record()
        e1.synchronize()
        best_ce = min(best_ce, e0.elapsed_time(e1))
    for _ in range(reps):
        torch.cuda.synchronize()
        e0.record()
        hs.hs_h2d_read(host.data_ptr(), dev.data_ptr(), nbytes, 0, torch.cuda.current_stream())
        e1.record()
        e1.synchronize()
        best_zc = min(best_zc, e0.elapsed_time(e1))
    ok = bool(torch.equal(dev[:4096].cpu(), host[:4096]))
    del host, dev
    ce = nbytes / best_ce / 1e6
    zc = nbytes / best_zc / 1e6
    return {"copy_engine_gbs": ce, "zero_copy_kernel_gbs": zc, "peak_gbs": max(ce, zc),
            "zero_copy_checked": ok, "bytes": nbytes}


def measure_hbm_peak(torch):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                v = float(json.load(f)["hbm_gbs"])
            return v, "MEASURED_PEAKS.json hbm_gbs (measured copy on this pool)"
        except (ValueError, KeyError, OSError):
            pass
    n = 1 << 30
    a = torch.empty(n, dtype=torch.uint8, device="cuda")
    b = torch.empty_like(a)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(5):
        e0.record()
        b.copy_(a)
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return 2 * n / best / 1e6, "device copy measured in this run (read + write bytes)"


# ---------------------------------------------------------------- ranks
def shard_requests(rank: int, batch: int):
    """Request ids of one rank: each rank owns its own block of B requests.

    The path partitions by request (every request owns its tables, stamps,
    buffer and host rows), so ranks share nothing on the data path."""
    return list(range(rank * batch, (rank + 1) * batch))


class RankOps:
    """Timing-only collectives over the ranks (none on the data path)."""

    def __init__(self, dist, device):
        self.dist = dist
        self.device = device

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def _reduce(self, x, op):
        if self.dist is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=op)
        return float(t.item())

    def max(self, x):
        return self._reduce(x, None if self.dist is None else self.dist.ReduceOp.MAX)

    def sum(self, x):
        return self._reduce(x, None if self.dist is None else self.dist.ReduceOp.SUM)


def _quantiles(xs):
    """min, 10 %, median, 90 %, max of the per-step times, and the means of the first and last tenth."""
    v = sorted(xs)
    n = len(v)
    k = max(1, n // 10)
    return {"min": v[0], "p10": v[n // 10], "p50": v[n // 2], "p90": v[(9 * n) // 10], "max": v[-1],
            "first_tenth_mean": sum(xs[:k]) / k, "last_tenth_mean": sum(xs[-k:]) / k}


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, dist):
    import torch
    from hierarchical_kv_cache_hs_gb300 import hs
    from hierarchical_kv_cache_hs_gb300 import tracegen as tg
    from hierarchical_kv_cache_hs_gb300.workload import GpuWorkload

    wl = tg.WORKLOADS[args.workload]
    mode = {"auto": hs.HS_COPY_AUTO, "fused": hs.HS_COPY_FUSED, "split": hs.HS_COPY_SPLIT,
            "cluster": hs.HS_COPY_CLUSTER}[args.copy_mode]
    hs.hs_set_host_pool_pages({"auto": hs.HS_POOL_PAGES_AUTO, "base": hs.HS_POOL_PAGES_BASE,
                               "huge": hs.HS_POOL_PAGES_HUGE}[args.pool_pages])
    total_steps = PRIME_STEPS + args.warmup + args.steps
    # Several layers: one launch for all of them, or one call per layer.
    one = args.layer_launch == "one" and wl.layers > 1
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    ops = RankOps(dist, dev)
    barrier, max_over_ranks, sum_over_ranks = ops.barrier, ops.max, ops.sum

    if args.no_peaks:
        peaks = {"copy_engine_gbs": None, "zero_copy_kernel_gbs": None, "peak_gbs": float("nan"),
                 "zero_copy_checked": None, "bytes": 0}
    else:
        peaks = measure_h2d_peak(torch, hs)
    hbm_gbs, hbm_src = measure_hbm_peak(torch)

    def measure(wl, want_profile=True, want_e2e=True, want_ce=False, one_launch=None):
        # Several layers: one launch for all of them, or one call per layer.
        one = (args.layer_launch == "one" and wl.layers > 1) if one_launch is None else one_launch
        w = GpuWorkload(wl, steps=total_steps, record=False, host_trace=want_e2e,
                        request_offset=shard_requests(rank, wl.B)[0], copy_mode=mode)
        stream = torch.cuda.Stream(device=dev)
        # The library's launch mode for this handle: one kernel (fused, or a
        # cluster of CTAs per request) or two (split).
        kind = hs.hs_launch_mode(w.handles[0].h)
        res = {"fused": kind != hs.HS_COPY_SPLIT, "cluster": kind == hs.HS_COPY_CLUSTER,
               "cluster_size": hs.hs_cluster_size(w.handles[0].h),
               "pool_pages": ("huge-page memory, cudaHostRegister"
                              if hs.hs_host_pool_pages(w.handles[0].h) == hs.HS_POOL_PAGES_HUGE
                              else "cudaHostAlloc")}
        try:
            def stats_sum(key):
                return sum(hs.hs_stats(h.h)[key] for h in w.handles)

            # --- device-resident timed pass -------------------------------
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            launches = 0
            misses_per_step = []
            with torch.cuda.stream(stream):
                for s in range(PRIME_STEPS + args.warmup):
                    w.launch_step(s, stream, one_launch=one)
                stream.synchronize()
                m0 = stats_sum("misses")
                i0 = stats_sum("inplace")
                barrier()
                torch.cuda.synchronize()
                t_wall0 = time.perf_counter()
                for i in range(args.steps):
                    s = PRIME_STEPS + args.warmup + i
                    flush.fill_(i & 0xFF)
                    starts[i].record(stream)
                    launches += w.launch_step(s, stream, one_launch=one)
                    ends[i].record(stream)
                torch.cuda.synchronize()
                barrier()
                t_wall = time.perf_counter() - t_wall0
            step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
            dev_ms = sum(step_ms)
            miss_rows = stats_sum("misses") - m0
            res.update(dev_ms=dev_ms, step_ms=step_ms, wall_s=t_wall, launches=launches,
                       miss_rows=miss_rows, inplace=stats_sum("inplace") - i0)

            # --- per-step miss counts + copy-kernel durations (second pass) ----
            if want_profile:
                w.reset()
                before = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
                after = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
                rs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
                copy_ms = []
                resolve_ms = []
                import numpy as np
                last = np.zeros(wl.B, dtype=np.int32)
                with torch.cuda.stream(stream):
                    for s in range(PRIME_STEPS + args.warmup):
                        w.launch_step(s, stream, one_launch=one)
                    for i in range(args.steps):
                        s = PRIME_STEPS + args.warmup + i
                        flush.fill_(i & 0xFF)
                        tot = 0
                        cms = rms = 0.0
                        if one:
                            # One launch covers every layer: time it whole.
                            before[i].record(stream)
                            w.launch_step(s, stream, one_launch=True)
                            after[i].record(stream)
                            stream.synchronize()
                            for h in w.handles:
                                hs.hs_stats(h.h, last)
                                tot += int(last.sum())
                            misses_per_step.append(tot)
                            copy_ms.append(before[i].elapsed_time(after[i]))
                            resolve_ms.append(0.0)
                            continue
                        for layer, h in enumerate(w.handles):
                            for e in (before[i], after[i], rs[i]):
                                e.record(stream)
                            hs.hs_profile_events(h.h, before[i], after[i])
                            if w.append_rows is not None:
                                hs.hs_append(h.h, w.append_rows[layer, s], stream)
                            rs[i].record(stream)
                            hs.hs_resolve(h.h, w.topk[layer, s], wl.K, w.out[layer], stream)
                            hs.hs_profile_events(h.h, None, None)
                            stream.synchronize()
                            hs.hs_stats(h.h, last)
                            tot += int(last.sum())
                            cms += before[i].elapsed_time(after[i])
                            rms += rs[i].elapsed_time(before[i])
                        misses_per_step.append(tot)
                        copy_ms.append(cms)
                        resolve_ms.append(rms)
                res.update(misses_per_step=misses_per_step, copy_ms=copy_ms, resolve_ms=resolve_ms)

            # --- copy-engine comparison variant (hs_resolve_ce) ------------
            if want_ce:
                w.reset()
                n_ce = min(args.steps, 30)
                with torch.cuda.stream(stream):
                    for s in range(PRIME_STEPS + args.warmup):
                        w.launch_step(s, stream)
                    ce_s = 0.0
                    for i in range(n_ce):
                        s = PRIME_STEPS + args.warmup + i
                        flush.fill_(i & 0xFF)
                        stream.synchronize()
                        t0 = time.perf_counter()
                        w.launch_step(s, stream, copy_engine=True)
                        stream.synchronize()
                        ce_s += time.perf_counter() - t0
                res.update(ce_s=ce_s, ce_steps=n_ce)

            # --- end to end through hs_resolve_host -----------------------
            if want_e2e:
                w.reset()
                out_host = torch.empty((wl.layers, wl.B, wl.K), dtype=torch.int32).pin_memory()
                with torch.cuda.stream(stream):
                    for s in range(PRIME_STEPS + args.warmup):
                        w.host_step(s, out_host, stream, one_launch=one)
                    e2e_s = 0.0
                    for i in range(args.steps):
                        s = PRIME_STEPS + args.warmup + i
                        flush.fill_(i & 0xFF)
                        stream.synchronize()
                        t0 = time.perf_counter()
                        w.host_step(s, out_host, stream, one_launch=one)
                        e2e_s += time.perf_counter() - t0
                res.update(e2e_s=e2e_s)
        finally:
            w.close()
        return res

    sampler = ClockSampler(dev.index, args.clocks_csv)
    main = measure(wl, want_e2e=not args.no_e2e, want_ce=not args.no_ce, one_launch=one)
    clocks = sampler.stop()

    def policy_sweep(wl):
        """Buffer size x eviction policy: the axes of the blog's miss-count figure."""
        out = {}
        w = GpuWorkload(wl, steps=total_steps, record=False, request_offset=shard_requests(rank, wl.B)[0],
                        copy_mode=mode)
        stream = torch.cuda.Stream(device=dev)
        try:
            for pname, pol in POLICIES:
                w.reset()
                for h in w.handles:
                    hs.hs_set_policy(h.h, pol)
                import numpy as np
                last = np.zeros(wl.B, dtype=np.int32)
                per_step = []
                e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
                e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
                with torch.cuda.stream(stream):
                    # Timed pass: launches queued ahead as in the main pass, so no
                    # host round trip falls inside a step's events.
                    for s in range(PRIME_STEPS + args.warmup):
                        w.launch_step(s, stream)
                    for i in range(args.steps):
                        s = PRIME_STEPS + args.warmup + i
                        flush.fill_(i & 0xFF)
                        e0[i].record(stream)
                        w.launch_step(s, stream)
                        e1[i].record(stream)
                    stream.synchronize()
                    ms = sum(a.elapsed_time(b) for a, b in zip(e0, e1))
                    # Counting pass over the same steps: per-step miss counts.
                    w.reset()
                    for h in w.handles:
                        hs.hs_set_policy(h.h, pol)
                    for s in range(PRIME_STEPS + args.warmup):
                        w.launch_step(s, stream)
                    for i in range(args.steps):
                        w.launch_step(PRIME_STEPS + args.warmup + i, stream)
                        tot = 0
                        for h in w.handles:
                            hs.hs_stats(h.h, last)
                            tot += int(last.sum())
                        per_step.append(tot)
                gbs = sum(per_step) * wl.row_bytes / (ms / 1e3) / 1e9
                out[pname] = {
                    "resolves_per_s": wl.B * wl.layers * args.steps / (ms / 1e3),
                    "ms_per_step": ms / args.steps,
                    "miss_row_gbs": gbs,
                    "miss_row_frac_of_h2d_peak": gbs / peaks["peak_gbs"],
                    "misses_per_step_mean": statistics.mean(per_step),
                    "misses_per_step": per_step,
                }
        finally:
            w.close()
        return out

    def miss_curve(base):
        """Misses per request per step against the buffer size, for each policy: the
        curve behind the blog's miss-count figure (buffer size x eviction policy), on the
        first MISS_CURVE_REQUESTS requests of the workload's trace (the generator keys each
        request's trace by its id, so they are the same requests as in the full run).
        Counting only; the steps are not timed."""
        import numpy as np
        B = min(MISS_CURVE_REQUESTS, base.B)
        curve = {"requests": B, "steps": args.steps, "buffer_slots": list(MISS_CURVE_SLOTS)}
        curve.update({pname: [] for pname, _ in POLICIES})
        stream = torch.cuda.Stream(device=dev)
        for S in MISS_CURVE_SLOTS:
            wl = base.with_(B=B, S=S, host_ratio=-(-base.cold // S))
            w = GpuWorkload(wl, steps=total_steps, record=False, copy_mode=mode)
            try:
                last = np.zeros(B, dtype=np.int32)
                for pname, pol in POLICIES:
                    w.reset()
                    for h in w.handles:
                        hs.hs_set_policy(h.h, pol)
                    misses = 0
                    with torch.cuda.stream(stream):
                        for s in range(PRIME_STEPS + args.warmup):
                            w.launch_step(s, stream)
                        for i in range(args.steps):
                            w.launch_step(PRIME_STEPS + args.warmup + i, stream)
                            hs.hs_stats(w.handles[0].h, last)
                            misses += int(last.sum())
                    curve[pname].append(misses / (B * args.steps))
            finally:
                w.close()
        return curve

    # Eviction policies of the sweep and the curve (random eviction keeps the
    # handles' default seed, 0).
    POLICIES = (("lru", hs.HS_POLICY_LRU), ("fifo", hs.HS_POLICY_FIFO), ("random", hs.HS_POLICY_RANDOM))
    sweep = {}
    curve = None
    if not args.no_sweep and args.workload == "b64_c64k_s4096":
        for name in ("b64_c64k_s4096", "b64_c64k_s2048"):
            sweep[name] = policy_sweep(tg.WORKLOADS[name])
        if rank == 0:
            curve = miss_curve(tg.WORKLOADS["b64_c64k_s4096"])

    def summarize(wl, res, one):
        """The metric, both rooflines and the end-to-end figure of one measured workload."""
        fused = res["fused"]
        units = wl.B * wl.layers * args.steps
        dev_s = max_over_ranks(res["dev_ms"] / 1e3)
        all_units = sum_over_ranks(units)
        value = all_units / dev_s
        miss_gbs = sum_over_ranks(res["miss_rows"] * wl.row_bytes) / dev_s / 1e9
        h2d_peak = peaks["peak_gbs"]
        # Roofline of the dominant kernel (the swap-in kernel, or the row copy in
        # split mode): algorithmic bytes are the miss rows (R bytes each) read over
        # the host link, per launch.
        copy_s = sum(res["copy_ms"]) / 1e3
        copy_gbs = (sum(res["misses_per_step"]) * wl.row_bytes) / copy_s / 1e9
        # Whole-step roofline: max(miss bytes / H2D peak, table bytes / HBM peak).
        t_roof = 0.0
        for m in res["misses_per_step"]:
            table = wl.layers * (wl.B * (16 * wl.K + 4 * wl.S)) + 16 * m
            t_roof += max(m * wl.row_bytes / (h2d_peak * 1e9), table / (hbm_gbs * 1e9))
        cl = res["cluster"] and not one
        kernel = ("hs_resolve_layers_kernel" if one else "hs_swapin_cluster_kernel" if cl
                  else "hs_resolve_kernel_fused" if fused else "hs_copy_kernel")
        traffic, host_link, traffic_src = dram_traffic(kernel, wl.name)
        e2e_value = all_units / max_over_ranks(res["e2e_s"]) if "e2e_s" in res else None
        out = {
            "value": value,
            "ms_per_step": res["dev_ms"] / args.steps,
            "miss_row_gbs": miss_gbs,
            "miss_row_frac_of_h2d_peak": miss_gbs / h2d_peak,
            "step_roofline": {"t_roof_ms_per_step": t_roof * 1e3 / args.steps,
                              "frac": t_roof / (res["dev_ms"] / 1e3),
                              "hbm_peak_gbs": hbm_gbs, "hbm_peak_source": hbm_src,
                              "table_bytes_per_resolve": "16K + 4S + 16m"},
            "roofline": {"bound": "h2d",
                         "kernel": ("hs_resolve_layers_kernel (every layer's resolve + row fetch, "
                                    "one grid)" if one else
                                    "hs_swapin_cluster_kernel (resolve + row fetch, a cluster of "
                                    "%d CTAs per request)" % res["cluster_size"] if cl else
                                    "hs_resolve_kernel<fused> (resolve + row fetch)" if fused
                                    else "hs_copy_kernel"),
                         "achieved": copy_gbs,
                         "peak": h2d_peak, "unit": "GB/s", "frac": copy_gbs / h2d_peak,
                         "traffic": traffic,
                         "traffic_host_link": host_link,
                         "traffic_source": traffic_src,
                         "peak_source": "measured in this run: max(1 GiB pinned->device "
                                        "cudaMemcpyAsync, 1 GiB zero-copy 128-bit read kernel)"},
            "kernel_ms_per_step": ({"swapin_fused": sum(res["copy_ms"]) / args.steps}
                                   if (fused or one) else
                                   {"copy": sum(res["copy_ms"]) / args.steps,
                                    "resolve": sum(res["resolve_ms"]) / args.steps}),
            "launch_mode": ("fused, all layers in one launch" if one else
                            "cluster of %d CTAs per request" % res["cluster_size"] if cl else
                            "fused" if fused else "split"),
            "host_pool": res["pool_pages"],
            "misses_per_step_mean": statistics.mean(res["misses_per_step"]),
            "inplace_per_step_mean": res["inplace"] / args.steps,
            "e2e": {"value": e2e_value, "unit": "resolves/s",
                    "h2d_bytes_per_step": wl.layers * wl.B * wl.K * 4,
                    "d2h_bytes_per_step": wl.layers * wl.B * wl.K * 4,
                    "api": ("hs_resolve_layers_host" if one else "hs_resolve_host") +
                           " (pinned host top-k in, host out_slot back, synchronised)"},
        }
        return out

    head = summarize(wl, main, one)
    line = {
        "metric": METRIC,
        "value": head["value"],
        "unit": "resolves/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int32",
        "data": "synthetic (seeded top-k traces and uniform random KV row bytes)",
        "config": _config(wl),
    }
    line.update({k: v for k, v in head.items() if k not in ("value", "ms_per_step")})
    line["h2d_peak"] = peaks
    line["misses_per_step"] = main["misses_per_step"]
    line["gpu_launches"] = main["launches"]
    line["clocks"] = clocks
    line["wall_s_timed_region"] = main["wall_s"]
    line["step_ms_quantiles"] = _quantiles(main["step_ms"])
    line["context"] = CONTEXT
    line["setup"] = ("each host pool is filled, then read once by the GPU (hs_h2d_read) before "
                     "the first step, as a long-lived serving pool is warm; the first 10 trace "
                     "steps and the warm-up steps run untimed")
    if args.overlap and rank == 0:
        line["layer_overlap"] = layer_overlap(args, torch, hs, tg, GpuWorkload, flush, dev)
    # The headline workload's default run includes it, beside the policy sweep.
    headline_default = not args.no_sweep and args.workload == "b64_c64k_s4096"
    if (args.overlap_compute or headline_default) and rank == 0 and world == 1:
        line["compute_overlap"] = compute_overlap(args, torch, hs, tg, GpuWorkload, wl)
    if "ce_s" in main:
        ce_value = wl.B * wl.layers * main["ce_steps"] / main["ce_s"]
        line["copy_engine_variant"] = {
            "api": "hs_resolve_ce: miss tokens read back, host-thread gather into pinned staging, "
                   "one cudaMemcpyAsync, device scatter (host wall time per step, synchronised)",
            "resolves_per_s": ce_value,
            "ms_per_step": main["ce_s"] * 1e3 / main["ce_steps"],
            "steps": main["ce_steps"],
            "faster": ("zero-copy (hs_resolve)" if head["value"] > ce_value
                       else "copy-engine (hs_resolve_ce)"),
        }
    if sweep:
        line["sweep"] = sweep
    if curve is not None:
        line["miss_curve"] = curve
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args, total_steps)

    # Every other workload, each at its own sizes, with the same steps and
    # warm-up: the parity-test workloads measured by the same passes.
    if not args.no_configs:
        per = {}
        for name in args.configs.split(","):
            if name == wl.name or not name:
                continue
            cw = tg.WORKLOADS[name]
            c_one = args.layer_launch == "one" and cw.layers > 1
            sampler = ClockSampler(dev.index)
            res = measure(cw, want_e2e=not args.no_e2e, one_launch=c_one)
            c_clocks = sampler.stop()
            entry = {"workload": _workload_desc(cw), "steps": args.steps, "warmup": args.warmup}
            entry.update(summarize(cw, res, c_one))
            entry["gpu_launches"] = res["launches"]
            entry["clocks"] = c_clocks
            entry["step_ms_quantiles"] = _quantiles(res["step_ms"])
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                entry["cpu_baseline"] = cpu_baseline(cw, args, total_steps, host_bytes=CONFIG_ORACLE_HOST_BYTES,
                                                     single_core=False)
            per[name] = entry
        line["configs"] = per
    return line


def compute_overlap(args, torch, hs, tg, GpuWorkload, wl):
    """The swap-in steps beside other work on another stream: bf16 4096^3 GEMMs
    (cuBLAS, standing in for a model's compute), about as many as take the
    steps' time.  Per launch setup: the steps alone, the GEMMs alone, both at
    once, and the share of the shorter one hidden, (alone + alone - both) /
    min(alone, alone).  One layer; the L2 is not flushed here."""
    prime, n = PRIME_STEPS, 30
    wl = wl.with_(layers=1)
    w = GpuWorkload(wl, steps=prime + n)
    a = torch.randn(4096, 4096, dtype=torch.bfloat16, device="cuda")
    c = torch.empty_like(a)
    sa, sb, main = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.current_stream()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def gemms(g, stream):
        with torch.cuda.stream(stream):
            for _ in range(g):
                torch.matmul(a, a, out=c)

    def prime_steps():
        w.reset()
        with torch.cuda.stream(sb):
            for s in range(prime):
                w.launch_step(s, sb)
        torch.cuda.synchronize()

    def steps(stream):
        with torch.cuda.stream(stream):
            for s in range(prime, prime + n):
                w.launch_step(s, stream)

    out = {"workload": _workload_desc(wl), "steps": n,
           "gemm": "torch.matmul bf16 4096 x 4096 x 4096 on another stream"}
    try:
        for _ in range(20):
            torch.matmul(a, a, out=c)
        e0, e1 = ev(), ev()
        e0.record(main)
        gemms(50, main)
        e1.record(main)
        torch.cuda.synchronize()
        t_one = e0.elapsed_time(e1) / 50
        g = None
        for tag, mode, ctas in (("default", hs.HS_COPY_AUTO, 0), ("fused", hs.HS_COPY_FUSED, 0),
                                ("split_48_copy_ctas", hs.HS_COPY_SPLIT, 48)):
            for h in w.handles:
                hs.hs_set_copy_mode(h.h, mode)
                hs.hs_set_copy_ctas(h.h, ctas)
            prime_steps()
            e0, e1 = ev(), ev()
            e0.record(sb)
            steps(sb)
            e1.record(sb)
            torch.cuda.synchronize()
            t_swap = e0.elapsed_time(e1)
            if g is None:
                g = max(1, int(round(t_swap / t_one)))
                out["gemms"] = g
            e0, e1 = ev(), ev()
            e0.record(sa)
            gemms(g, sa)
            e1.record(sa)
            torch.cuda.synchronize()
            t_gemm = e0.elapsed_time(e1)
            prime_steps()
            e0, e1 = ev(), ev()
            e0.record(main)
            sa.wait_stream(main)
            sb.wait_stream(main)
            gemms(g, sa)
            steps(sb)
            main.wait_stream(sa)
            main.wait_stream(sb)
            e1.record(main)
            torch.cuda.synchronize()
            t_both = e0.elapsed_time(e1)
            out[tag] = {"swapin_ms": t_swap, "gemm_ms": t_gemm, "both_ms": t_both,
                        "hidden": (t_swap + t_gemm - t_both) / min(t_swap, t_gemm)}
    finally:
        w.close()
    return out


def layer_overlap(args, torch, hs, tg, GpuWorkload, flush, dev):
    """Independent layers: one call per layer on one stream, one stream per layer,
    or all layers in one launch."""
    wl = tg.WORKLOADS["b64_c128k_l4_tail4096"]
    steps = PRIME_STEPS + args.warmup + args.steps
    w = GpuWorkload(wl, steps=steps)
    out = {"workload": _workload_desc(wl)}
    try:
        main = torch.cuda.Stream(device=dev)
        lstreams = [torch.cuda.Stream(device=dev) for _ in range(wl.layers)]
        for name, ls, one in (("one_stream", None, False), ("stream_per_layer", lstreams, False),
                              ("one_launch", None, True)):
            w.reset()
            ms = 0.0
            with torch.cuda.stream(main):
                for s in range(PRIME_STEPS + args.warmup):
                    w.launch_step(s, main, layer_streams=ls, one_launch=one)
                for i in range(args.steps):
                    s = PRIME_STEPS + args.warmup + i
                    flush.fill_(i & 0xFF)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(main)
                    w.launch_step(s, main, layer_streams=ls, one_launch=one)
                    e1.record(main)
                    e1.synchronize()
                    ms += e0.elapsed_time(e1)
            out[name] = {"resolves_per_s": wl.B * wl.layers * args.steps / (ms / 1e3),
                         "ms_per_step": ms / args.steps}
        misses = sum(hs.hs_stats(h.h)["misses"] for h in w.handles)
        out["misses_last_pass"] = misses
    finally:
        w.close()
    return out


# ---------------------------------------------------------------- CPU oracle
ORACLE_HOST_BYTES = 8 << 30  # host rows the oracle legs may hold at once
CONFIG_ORACLE_HOST_BYTES = 1 << 30  # the same for the other workloads' legs
# The five workloads, in the order of the pages' configurations; the bench
# workload is the headline line, the others go under "configs".
CONFIG_WORKLOADS = ("tiny_b1_c8k", "b32_c32k_s4096", "b64_c64k_s4096", "b64_c64k_s2048",
                    "b256_c32k_grow_tail512", "b64_c128k_l4_tail4096")


def _oracle_sample(wl, host_bytes=ORACLE_HOST_BYTES):
    """Requests the oracle legs replay: all of them, or the first n whose host
    rows (every layer) fit in host_bytes."""
    per_request = wl.layers * wl.cold * wl.row_bytes
    n = max(1, min(wl.B, host_bytes // max(per_request, 1)))
    return list(range(n))


def _oracle_requests(wl, total_steps, requests, threads, time_from_step):
    """Replay the trace on the CPU oracle for the given requests of every
    layer, appending each step's new token first on a growing context; returns
    seconds spent on steps >= time_from_step."""
    import oracle
    from hierarchical_kv_cache_hs_gb300 import tracegen as tg
    jobs = [(layer, i) for layer in range(wl.layers) for i in range(len(requests))]
    traces = [tg.topk_trace(wl, layer=layer, steps=total_steps, requests=requests)
              for layer in range(wl.layers)]
    hosts, appends = {}, {}

    def prep(job):
        layer, i = job
        hosts[job] = tg.rows(wl, layer, requests[i], 0, wl.cold)
        if wl.grow:
            appends[job] = tg.rows(wl, layer, requests[i], wl.len0, total_steps)

    oracle.parallel_map(prep, jobs, threads)
    length = wl.len0 if (wl.grow or wl.sliding) else wl.C
    states = {job: oracle.RequestState(wl.C, wl.S, wl.T, wl.row_bytes, length, sliding=wl.sliding)
              for job in jobs}
    from concurrent.futures import ThreadPoolExecutor

    elapsed = 0.0
    with ThreadPoolExecutor(threads) as ex:
        for s in range(total_steps):
            def run(job, s=s):
                st = states[job]
                if wl.grow:
                    st.append(appends[job][s], hosts[job])
                st.resolve(hosts[job], traces[job[0]][s, job[1]], s + 1)
            t0 = time.perf_counter()
            list(ex.map(run, jobs))
            if s >= time_from_step:
                elapsed += time.perf_counter() - t0
    return elapsed


def _sample_desc(wl, requests):
    who = "all %d requests" % wl.B if len(requests) == wl.B else "requests 0-%d of %d" % (
        len(requests) - 1, wl.B)
    layers = "" if wl.layers == 1 else " of each of the %d layers" % wl.layers
    grow = ", each step's new token appended first" if wl.grow else ""
    return who + layers + grow


def cpu_baseline(wl, args, total_steps, host_bytes=ORACLE_HOST_BYTES, single_core=True):
    """The oracle as it stands on every host core (and on one), over a bounded
    sample of the workload's requests."""
    cores = _cores()
    from_step = PRIME_STEPS + args.warmup
    reqs = _oracle_sample(wl, host_bytes)
    secs = _oracle_requests(wl, total_steps, reqs, cores, from_step)
    n = len(reqs) * wl.layers * (total_steps - from_step)
    out = {"value": n / secs, "unit": "resolves/s", "cores": cores, "kind": "oracle",
           "sample": "the timed steps of the same trace, %s, one request per thread per step, "
                     "after replaying the untimed prefix" % _sample_desc(wl, reqs)}
    if single_core:
        # The same on one core, over the first few requests.
        reqs1 = reqs[:min(8, len(reqs))]
        secs1 = _oracle_requests(wl, total_steps, reqs1, 1, from_step)
        out["single_core"] = {"value": len(reqs1) * wl.layers * (total_steps - from_step) / secs1,
                              "unit": "resolves/s", "cores": 1,
                              "sample": "the same timed steps, %s" % _sample_desc(wl, reqs1)}
    return out


def run_reference(args):
    from hierarchical_kv_cache_hs_gb300 import tracegen as tg
    wl = tg.WORKLOADS[args.workload]
    total_steps = PRIME_STEPS + args.warmup + args.steps
    cores = _cores()
    reqs = _oracle_sample(wl)
    secs = _oracle_requests(wl, total_steps, reqs, cores, PRIME_STEPS + args.warmup)
    units = len(reqs) * wl.layers * args.steps
    value = units / secs
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "resolves/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": secs * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int32",
        "data": "synthetic (seeded top-k traces and uniform random KV row bytes)",
        "config": _config(wl),
        "cpu_baseline": {"value": value, "unit": "resolves/s", "cores": cores, "kind": "oracle",
                         "sample": "every timed step of the workload, %s, one request per thread"
                                   % _sample_desc(wl, reqs)},
        "e2e": {"value": value, "unit": "resolves/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=180)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="b64_c64k_s4096")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (the \"configs\" key)")
    ap.add_argument("--configs", default=",".join(CONFIG_WORKLOADS),
                    help="comma-separated workloads measured under \"configs\" besides --workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-peaks", action="store_true",
                    help="skip the 1 GiB link-peak measurement (profiling runs; no roofline fraction)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer pass")
    ap.add_argument("--no-ce", action="store_true", help="skip the copy-engine comparison variant")
    ap.add_argument("--layer-launch", choices=["one", "loop"], default="one",
                    help="several layers: all in one launch (hs_resolve_layers) or one call per layer")
    ap.add_argument("--clocks-csv", default=None,
                    help="also write the nvidia-smi clock samples of the timed region to this file")
    ap.add_argument("--overlap", action="store_true",
                    help="also time the 4-layer, 128K-context workload with its layers on one "
                         "stream and on one stream per layer")
    ap.add_argument("--copy-mode", choices=["auto", "fused", "split", "cluster"], default="auto",
                    help="launch mode of the step (identical results; see hs_set_copy_mode)")
    ap.add_argument("--overlap-compute", action="store_true",
                    help="time the step beside bf16 GEMMs on another stream, per launch setup "
                         "(on by default for the headline workload; --no-sweep turns it off)")
    ap.add_argument("--pool-pages", choices=["auto", "base", "huge"], default="auto",
                    help="host pool placement (identical results; see hs_set_host_pool_pages)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    from hierarchical_kv_cache_hs_gb300 import build
    if rank == 0:
        build.build_all()
    if dist is not None:
        dist.barrier()
    line = run_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
