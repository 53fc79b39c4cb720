"""Benchmark: int32 TopK (k = 20) over 1e8 elements on one GB300, plus the
row TopK workload, printed as ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one topk_i32 call over the resident 1e8-element input (uniform over
the full int32 range, seed 2), the shape of the TopK pages' headline
benchmark ("CUDA parallel optimisation: TopK, shared memory and two-stage
reduction", section 4.1: 1e8 ints, top 20).  The input (400 MB) is larger
than the 129 MB L2, so no flush is needed between steps.

Under torchrun every rank runs its own replica of the workload on its own
GPU (independent problems, weak scaling); rank 0 prints the line with the
elapsed time of the slowest rank.

--impl reference times the CPU oracle (single-threaded std::sort, the
definition the GPU result is checked against) on bounded samples of the same
workload; it is the slow reference arm, not a target.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

WORKLOAD = "i32_uniform_1e8"
K_TOP = 20
METRIC = "TopK Gelem/s and achieved HBM GB/s (% of ~8 TB/s) at 1e8 int32, k=20"
UNIT = "Gelem/s"


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


KERNEL_SOURCES = {
    "topk_i32_stream_kernel": ("topk_i32.cu", "topk_device.cuh", "topk_internal.h"),
    "topk_rows_stream_kernel": ("topk_rows.cu", "topk_device.cuh", "topk_internal.h", "topk_sortnet.cuh"),
    "radix_filter_kernel": ("topk_radix.cu", "topk_device.cuh", "topk_internal.h", "topk_sortnet.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources a kernel is built from (its .cu and shared headers)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "topk_selection_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary,
    if it was taken on the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        e = rec[f"{kernel}@{workload}"]
        if e.get("source_hash") == kernel_source_hash(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples, tagged with host receive times."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not win:  # a very short timed region: take the samples nearest to it
            win = [p for (t, p) in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        smax = [num(p[1]) for p in win if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(win)}


class Timer:
    """CUDA-event timing of library calls on one stream.

    single(fn): one call alone, device time -- the previous work on the stream has
    finished and L2 holds none of the input (a 512 MiB buffer is read
    first, outside the timed region: reading leaves clean lines in L2, so no
    write-back of the flush lands in the timed call); the median over `reps`
    calls.
    pipelined(fn): `reps` calls back to back between two events; the mean per
    call.  Consecutive calls may overlap (a call starts streaming its input
    while the previous one's last block finishes), which is what a stream of
    independent TopK calls sees."""

    def __init__(self, dev, stream):
        self.stream = stream
        self.flush_buf = torch.empty(128 << 20, dtype=torch.int32, device=dev)  # 512 MiB
        self.flips = 0

    def flush(self):
        self.flips += 1
        self.sink = torch.sum(self.flush_buf, dtype=torch.int32)

    def single(self, fn, reps):
        ts = []
        for _ in range(reps):
            self.flush()
            # Keep the stream busy until the call below is enqueued, so the
            # first event marks the GPU reaching the call, not the host
            # entering it (host-side API time is in `e2e`).
            torch.cuda._sleep(100_000)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            fn()
            e1.record(self.stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    def pipelined(self, fn, reps):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for _ in range(reps):
            fn()
        e1.record(self.stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps


def run_ours(args, world, rank, local):
    import topk_selection_gb300 as tk

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n = synth.I32_WORKLOADS[WORKLOAD][1]
    x_host = torch.empty(n, dtype=torch.int32).pin_memory()
    synth.i32_workload(WORKLOAD, out=x_host.numpy())
    x = x_host.to(dev)
    out = torch.empty(K_TOP, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    s_handle = stream.cuda_stream

    def step():
        rc = tk.topk_i32_ptr(x.data_ptr(), n, K_TOP, out.data_ptr(), s_handle)
        if rc != 0:
            raise tk.TopKError(rc, "topk_i32")

    sampler = ClockSampler(local)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    time.sleep(0.2)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = tk.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier(world)
    launches = tk.launch_count() - launches0
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, world)
    sampler.stop()
    clocks = sampler.summary(w0, w1)
    result = out.cpu().numpy().copy()

    timer = Timer(dev, stream)
    peak, peak_kind = load_peaks()
    # The same call alone: what one caller making one call sees.
    single_us = timer.single(step, 50)

    extra = {}
    configs = {}
    if not args.skip_rows:
        configs, sweep = run_configs(tk, dev, stream, timer, x_host, x, peak, single_us, ms / args.steps * 1e3)
        extra["midk_sweep"] = sweep
        extra["rows_f32"] = run_rows(tk, dev, stream, args, timer, peak, configs)
        extra["large_k"] = run_large_k(tk, x, stream, args, timer)
        extra["noalloc"] = run_noalloc(tk, x, stream, timer, peak)
        extra["keys"] = run_keys(tk, x, stream, timer, peak)
        extra["reduce"] = run_reduce(tk, x, stream, args)
        extra["items"] = run_items(tk, dev, stream, args)
        extra["sort"] = run_sort(tk, x, stream, args)

    # End to end through the C ABI with host buffers: the library copies the
    # pinned input to the device, selects, and copies the k results back.
    out_host = torch.empty(K_TOP, dtype=torch.int32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    tk.topk_i32_ptr(x_host.data_ptr(), n, K_TOP, out_host.data_ptr(), s_handle)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        rc = tk.topk_i32_ptr(x_host.data_ptr(), n, K_TOP, out_host.data_ptr(), s_handle)
        if rc != 0:
            raise tk.TopKError(rc, "topk_i32 (host buffers)")
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    barrier(world)
    e2e_ok = bool(np.array_equal(out_host.numpy(), result))

    if rank != 0:
        return None

    total = n * world
    sec_per_step = ms_max / 1e3 / args.steps
    value = total * args.steps / (ms_max / 1e3) / 1e9
    kernel_s = ms / 1e3 / args.steps  # one launch per step on this stream
    achieved = 4.0 * n / kernel_s / 1e9
    single_gbs = 4.0 * n / (single_us / 1e6) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(sec_per_step * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int32",
        "data": "synthetic: SplitMix64 uniform int32, seed 2, generated on the host",
        "config": {"workload": "int32 TopK, N=1e8 uniform full range (seed 2), k=20, output sorted descending",
                   "n": n, "k": K_TOP, "parallelism": f"replicas x{world}",
                   "l2": "input 400 MB > 129 MB L2; no flush between steps"},
        "gbs": round(achieved, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "traffic": recorded_traffic("topk_i32_stream_kernel", WORKLOAD),
                     "kernel": "topk_i32_stream_kernel<1,1> (k<=32)", "algorithmic_bytes_per_launch": 4 * n,
                     "timing": "CUDA events on the launching stream around the timed steps; one launch per step; "
                               "back-to-back launches overlap (each streams while the previous one finishes)",
                     "single_call": {"us": round(single_us, 2), "achieved": round(single_gbs, 1),
                                     "frac": round(single_gbs / peak, 4),
                                     "timing": "one call alone after an L2 flush; median of 50"}},
        "e2e": {"value": round(total * e2e_steps / e2e_s / 1e9, 4), "unit": UNIT,
                "h2d_bytes_per_step": 4 * n, "d2h_bytes_per_step": 4 * K_TOP,
                "steps": e2e_steps, "matches_device_result": e2e_ok},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    line.update(extra)
    if not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline_leg(x_host.numpy(), result)
    if configs:
        line["configs"] = configs
    return line


def _frac(nbytes, us, peak):
    return round(nbytes / (us / 1e6) / 1e9 / peak, 3)


def run_configs(tk, dev, stream, timer, x_host_1e8, x_1e8, peak, c3_single_us, c3_pipe_us):
    """Every int32 configuration of the TopK benchmark table (2^20, 1e7,
    1e8, 1e9 x three inputs; TopK page section 4.1) as a single call and in a
    stream of calls, each result checked exactly against the oracle (full
    sort up to 1e7, the oracle's one-pass checker above)."""
    import oracle

    h = stream.cuda_stream
    res = {}

    def entry(xd, xh, n, k, reps_single, reps_pipe, exact_full):
        o = torch.empty(k, dtype=torch.int32, device=dev)

        def call():
            rc = tk.topk_i32_ptr(xd.data_ptr(), n, k, o.data_ptr(), h)
            if rc != 0:
                raise tk.TopKError(rc, f"topk_i32 n={n} k={k}")

        su = timer.single(call, reps_single)
        pu = timer.pipelined(call, reps_pipe)
        got = o.cpu().numpy()
        ok = bool(np.array_equal(got, oracle.topk_i32(xh, k))) if exact_full else bool(oracle.check_topk_i32(xh, k, got))
        return su, pu, ok

    for name, wl, ks in (("C1", "i32_uniform_2p20", (20,)), ("C2", "i32_uniform_1e7", (20, 100))):
        xh = synth.i32_workload(wl)
        xd = torch.from_numpy(xh).to(dev)
        for k in ks:
            su, pu, ok = entry(xd, xh, xh.size, k, 50, 200, True)
            res[f"{name}_k{k}"] = {"single_us": round(su, 2), "pipe_us": round(pu, 2), "ok": ok}
        del xd
    xh = x_host_1e8.numpy()
    ok20 = bool(oracle.check_topk_i32(xh, 20, tk.topk_i32(x_1e8, 20).cpu().numpy()))
    res["C3_k20"] = {"single_us": round(c3_single_us, 2), "pipe_us": round(c3_pipe_us, 2),
                     "frac_single": _frac(4e8, c3_single_us, peak), "frac_pipe": _frac(4e8, c3_pipe_us, peak),
                     "ok": ok20}
    su, pu, ok = entry(x_1e8, xh, xh.size, 1, 30, 50, False)
    res["C3_k1"] = {"single_us": round(su, 2), "pipe_us": round(pu, 2), "frac_single": _frac(4e8, su, peak),
                    "frac_pipe": _frac(4e8, pu, peak), "ok": ok}

    # 1e9: one pinned host buffer and one device buffer serve the three inputs.
    n9 = 10**9
    xh9 = torch.empty(n9, dtype=torch.int32).pin_memory()
    xd9 = torch.empty(n9, dtype=torch.int32, device=dev)
    for name, wl in (("C4a_uniform", "i32_uniform_1e9"), ("C4b_ascending", "i32_ascending_1e9"),
                     ("C4c_dup1000", "i32_dup1000_1e9")):
        synth.i32_workload(wl, out=xh9.numpy())
        xd9.copy_(xh9)
        su, pu, ok = entry(xd9, xh9.numpy(), n9, 20, 10, 10, False)
        res[name] = {"single_us": round(su, 1), "pipe_us": round(pu, 1), "frac_single": _frac(4e9, su, peak),
                     "frac_pipe": _frac(4e9, pu, peak), "ok": ok}
    del xd9, xh9
    torch.cuda.empty_cache()

    # Mid-size inputs at 20 <= k <= 128, single calls.
    sweep = {}
    for n in (300_000, 1 << 20, 10**7):
        xh = synth.i32_uniform(n, 7)
        xd = torch.from_numpy(xh).to(dev)
        for k in (20, 64, 100, 128):
            o = torch.empty(k, dtype=torch.int32, device=dev)

            def call():
                rc = tk.topk_i32_ptr(xd.data_ptr(), n, k, o.data_ptr(), h)
                if rc != 0:
                    raise tk.TopKError(rc, "topk_i32 (sweep)")

            su = timer.single(call, 20)
            ok = bool(np.array_equal(o.cpu().numpy(), oracle.topk_i32(xh, k)))
            sweep[f"n{n}_k{k}"] = {"single_us": round(su, 2), "ok": ok}
        del xd
    sweep["workload"] = "int32 uniform full range (seed 7), single calls after an L2 flush, median of 20"
    return res, sweep


def run_rows(tk, dev, stream, args, timer, peak, configs):
    """The batched float32 row TopK with indices (4096 x 32768, k = 64), on
    the tied rows (1% of each row overwritten by the row maximum, seed 5) and
    on the same rows without the ties; one call alone and a stream of calls.
    Parity: the oracle on 32 sampled rows of each result, bit for bit."""
    import oracle

    w = synth.ROWS_WORKLOAD
    rows, cols, k = w["rows"], w["cols"], w["k"]
    xh = torch.empty(rows * cols, dtype=torch.float32).pin_memory()
    vals = torch.empty(rows, k, dtype=torch.float32, device=dev)
    idx = torch.empty(rows, k, dtype=torch.int32, device=dev)
    h = stream.cuda_stream
    nbytes = rows * cols * 4 + rows * k * 8
    res = {}
    for name, tied in (("tied", True), ("untied", False)):
        if tied:
            synth.f32_rows_tied(rows, cols, w["seed"], w["tie_frac"], out=xh.numpy())
        else:
            synth.f32_rows_normal(rows, cols, w["seed"], out=xh.numpy())
        x = xh.to(dev)

        def step():
            rc = tk.topk_rows_f32_ptr(x.data_ptr(), rows, cols, k, vals.data_ptr(), idx.data_ptr(), h)
            if rc != 0:
                raise tk.TopKError(rc, "topk_rows_f32")

        for _ in range(5):
            step()
        torch.cuda.synchronize()
        su = timer.single(step, 30)
        pu = timer.pipelined(step, max(10, min(200, args.steps // 20)))
        xr = xh.numpy().reshape(rows, cols)
        sample = np.arange(0, rows, rows // 32)
        ev, ei = oracle.topk_rows_f32(xr[sample], k)
        ok = bool(np.array_equal(idx.cpu().numpy()[sample], ei)) and \
            bool(np.array_equal(vals.cpu().numpy()[sample].view(np.uint32), ev.view(np.uint32)))
        res[name] = {"single_us": round(su, 2), "pipe_us": round(pu, 2),
                     "value_single": round(rows * cols / (su / 1e6) / 1e9, 3), "unit": UNIT,
                     "roofline": {"bound": "hbm", "peak": peak, "unit": "GB/s",
                                  "achieved_single": round(nbytes / (su / 1e6) / 1e9, 1),
                                  "frac_single": _frac(nbytes, su, peak),
                                  "achieved_pipe": round(nbytes / (pu / 1e6) / 1e9, 1),
                                  "frac_pipe": _frac(nbytes, pu, peak),
                                  "kernel": "topk_rows_stream_kernel<2> (k<=64)",
                                  "algorithmic_bytes_per_launch": nbytes,
                                  "traffic": recorded_traffic("topk_rows_stream_kernel", "rows_4096x32768_k64_tied")
                                  if tied else None},
                     "parity_32_rows": ok}
        configs[f"C5_{name}"] = {"single_us": round(su, 1), "pipe_us": round(pu, 1),
                                 "frac_single": _frac(nbytes, su, peak), "frac_pipe": _frac(nbytes, pu, peak),
                                 "ok": ok}
        if not tied:
            # The same rows at k above 128 (one block per row, radix-select cuts).
            for kb in (129, 1024):
                vb = torch.empty(rows, kb, dtype=torch.float32, device=dev)
                ib = torch.empty(rows, kb, dtype=torch.int32, device=dev)

                def stepb():
                    rc = tk.topk_rows_f32_ptr(x.data_ptr(), rows, cols, kb, vb.data_ptr(), ib.data_ptr(), h)
                    if rc != 0:
                        raise tk.TopKError(rc, "topk_rows_f32 (large k)")

                stepb()
                sub = timer.single(stepb, 5)
                pub = timer.pipelined(stepb, 5)
                evb, eib = oracle.topk_rows_f32(xr[sample[:8]], kb)
                okb = bool(np.array_equal(ib.cpu().numpy()[sample[:8]], eib))
                nb = rows * cols * 4 + rows * kb * 8
                res[f"untied_k{kb}"] = {"single_us": round(sub, 1), "pipe_us": round(pub, 1),
                                        "frac_single": _frac(nb, sub, peak), "frac_pipe": _frac(nb, pub, peak),
                                        "parity_8_rows": okb}
                del vb, ib
        del x
    res["workload"] = "fp32 rows 4096x32768 N(0,1) seed 5, tied: 1% of each row set to the row max; k=64"
    return res


LARGE_K = (1000, 32768)


def run_large_k(tk, x, stream, args, timer):
    """topk_i32 with k above the streaming plan's limit (the radix-select
    plan: sample, filter pass, cluster select, range sort) on the 1e8 input
    already on the device.  The roofline counts one read of the input."""
    n = x.numel()
    peak, _ = load_peaks()
    h = stream.cuda_stream
    res = {}
    for k in LARGE_K:
        out = torch.empty(k, dtype=torch.int32, device=x.device)

        def step():
            rc = tk.topk_i32_ptr(x.data_ptr(), n, k, out.data_ptr(), h)
            if rc != 0:
                raise tk.TopKError(rc, "topk_i32 (large k)")

        for _ in range(5):
            step()
        torch.cuda.synchronize()
        steps = max(10, min(200, args.steps // 20))
        l0 = tk.launch_count()
        pu = timer.pipelined(step, steps)
        launches = (tk.launch_count() - l0) // (steps + 1)
        su = timer.single(step, 20)
        res[f"k{k}"] = {"single_us": round(su, 2), "pipe_us": round(pu, 2),
                        "value_pipe": round(n / (pu / 1e6) / 1e9, 3), "unit": UNIT,
                        "launches_per_call": launches,
                        "roofline": {"bound": "hbm", "peak": peak, "unit": "GB/s",
                                     "frac_single": _frac(4 * n, su, peak), "frac_pipe": _frac(4 * n, pu, peak),
                                     "algorithmic_bytes_per_launch": 4 * n,
                                     "kernel": "whole plan (dominant kernel: radix_filter_kernel)",
                                     "traffic_dominant_kernel": recorded_traffic("radix_filter_kernel",
                                                                                 "i32_uniform_1e8_k1000")}}
    res["workload"] = "int32 TopK, N=1e8 uniform full range (seed 2), k in (1000, 32768), sorted descending"
    return res


def run_keys(tk, x, stream, timer, peak):
    """topk_u32 and topk_f32 on the 1e8 input's bits (uniform uint32 keys;
    float32 bit patterns, half negative, ~0.4% NaN), and topk_i32 at
    k = 131072 (the large-k plan with the LSD sort ordering the answer)."""
    n = x.numel()
    h = stream.cuda_stream
    xf = x.view(torch.float32)
    res = {}
    for name, fn, src, k in (("u32_k20", tk.topk_u32_ptr, x, 20), ("f32_k20", tk.topk_f32_ptr, xf, 20),
                             ("f32_k1000", tk.topk_f32_ptr, xf, 1000), ("i32_k131072", tk.topk_i32_ptr, x, 131072)):
        out = torch.empty(k, dtype=torch.int32, device=x.device)

        def step():
            rc = fn(src.data_ptr(), n, k, out.data_ptr(), h)
            if rc != 0:
                raise tk.TopKError(rc, name)

        step()
        su = timer.single(step, 20)
        pu = timer.pipelined(step, 20)
        res[name] = {"single_us": round(su, 2), "pipe_us": round(pu, 2), "frac_single": _frac(4 * n, su, peak),
                     "frac_pipe": _frac(4 * n, pu, peak)}
    res["workload"] = "N=1e8 words of the uniform int32 input (seed 2) read as uint32 / float32 bits"
    return res


def run_noalloc(tk, x, stream, timer, peak):
    """topk_i32_noalloc (scratch in a fixed 1 MiB device array, so a smaller
    grid for k <= 128) next to topk_i32 on the 1e8 input, k = 20."""
    import ctypes

    f = tk._lib.topk_i32_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    n = x.numel()
    out = torch.empty(K_TOP, dtype=torch.int32, device=x.device)
    h = stream.cuda_stream

    def step():
        rc = f(x.data_ptr(), n, K_TOP, out.data_ptr(), h)
        if rc != 0:
            raise tk.TopKError(rc, "topk_i32_noalloc")

    step()
    su = timer.single(step, 30)
    pu = timer.pipelined(step, 20)
    return {"single_us": round(su, 2), "pipe_us": round(pu, 2), "frac_single": _frac(4 * n, su, peak),
            "frac_pipe": _frac(4 * n, pu, peak),
            "workload": "topk_i32_noalloc, N=1e8 uniform (seed 2), k=20"}


def run_reduce(tk, x, stream, args):
    """topk_reduce_i32 (sum) on the 1e8 int32 input and topk_reduce_f32 (sum)
    on a float32 array of the same size; one launch per call, 4 bytes read
    per element."""
    n = x.numel()
    peak, _ = load_peaks()
    h = stream.cuda_stream
    xf = (x.to(torch.float64) * 2.0 ** -31).to(torch.float32)
    res = {}
    for name, t, is_float, odt in (("i32_sum", x, False, torch.int64), ("f32_sum", xf, True, torch.float64)):
        out = torch.empty(1, dtype=odt, device=x.device)

        def step():
            rc = tk.reduce_ptr(t.data_ptr(), n, is_float, 0, out.data_ptr(), h)
            if rc != 0:
                raise tk.TopKError(rc, "topk_reduce")

        for _ in range(5):
            step()
        torch.cuda.synchronize()
        steps = max(10, min(200, args.steps // 20))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / steps
        gbs = 4.0 * n / (ms / 1e3) / 1e9
        res[name] = {"steps": steps, "ms_per_step": round(ms, 5), "value": round(n / (ms / 1e3) / 1e9, 3),
                     "unit": UNIT,
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                                  "frac": round(gbs / peak, 4), "algorithmic_bytes_per_launch": 4 * n,
                                  "kernel": "reduce_kernel (one launch per call)"}}
    del xf
    res["workload"] = "sum of N=1e8 int32 (seed 2) and of the same values scaled to float32"
    return res


def run_items(tk, dev, stream, args):
    """topk_items_f32 on N=1e8 N(0,1) scores (seed 2), k=64, item = position:
    without a filter (4 bytes read per element) and with a keep mask of about
    half the positions (score + mask = 5 bytes per element at least)."""
    n, k = 10**8, 64
    peak, _ = load_peaks()
    h = stream.cuda_stream
    sh = torch.empty(n, dtype=torch.float32).pin_memory()
    synth.f32_normal(n, 2, out=sh.numpy())
    sc = sh.to(dev)
    mh = torch.from_numpy((synth.i32_uniform(n, 3) & 1).astype(np.uint8))
    keep = mh.to(dev)
    out_s = torch.empty(k, dtype=torch.float32, device=dev)
    out_i = torch.empty(k, dtype=torch.int64, device=dev)
    res = {}
    for name, kp, bytes_per in (("no_filter", None, 4), ("keep_half", keep, 5)):
        def step():
            rc = tk.topk_items_f32_ptr(sc.data_ptr(), 0, kp.data_ptr() if kp is not None else 0, n, k,
                                       out_s.data_ptr(), out_i.data_ptr(), 0, h)
            if rc != 0:
                raise tk.TopKError(rc, "topk_items_f32")

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        steps = max(5, min(100, args.steps // 40))
        l0 = tk.launch_count()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / steps
        gbs = bytes_per * n / (ms / 1e3) / 1e9
        res[name] = {"steps": steps, "ms_per_step": round(ms, 5), "value": round(n / (ms / 1e3) / 1e9, 3),
                     "unit": UNIT, "launches_per_step": (tk.launch_count() - l0) // steps,
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                                  "frac": round(gbs / peak, 4), "algorithmic_bytes_per_launch": bytes_per * n,
                                  "kernel": "whole call (dominant kernel: topk_rows_stream_kernel, level 1)"}}
    del sc, keep
    res["workload"] = "float32 N(0,1) scores N=1e8 (seed 2), k=64, items = positions; keep = low bit of a uniform int32 stream (seed 3)"
    return res


def run_sort(tk, x, stream, args):
    """topk_sort_u32 on the 1e8 input's bits as uint32 keys, keys only and
    with uint32 values (positions).  Algorithmic traffic: the histogram pass
    reads 4 bytes per key and each of the four digit passes reads and writes
    4 (keys) or 8 (pairs) bytes per key: 36 or 68 bytes per key."""
    n = x.numel()
    peak, _ = load_peaks()
    h = stream.cuda_stream
    vals = torch.arange(n, dtype=torch.int32, device=x.device)
    ko = torch.empty_like(x)
    vo = torch.empty_like(vals)
    res = {}
    for name, with_vals, bytes_per in (("keys", False, 36), ("pairs", True, 68)):
        def step():
            rc = tk.sort_u32_ptr(x.data_ptr(), vals.data_ptr() if with_vals else 0, n, ko.data_ptr(),
                                 vo.data_ptr() if with_vals else 0, h)
            if rc != 0:
                raise tk.TopKError(rc, "topk_sort_u32")

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        steps = max(5, min(50, args.steps // 100))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / steps
        gbs = bytes_per * n / (ms / 1e3) / 1e9
        res[name] = {"steps": steps, "ms_per_step": round(ms, 4), "value": round(n / (ms / 1e3) / 1e9, 3),
                     "unit": "Gkeys/s",
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                                  "frac": round(gbs / peak, 4), "algorithmic_bytes_per_launch": bytes_per * n,
                                  "kernel": "whole sort (5 launches; dominant: sort_pass_kernel)"}}
    del vals, ko, vo
    res["workload"] = "uint32 keys = bits of the N=1e8 uniform int32 input (seed 2); values = positions"
    return res


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def cpu_baseline_leg(x: np.ndarray, gpu_result: np.ndarray):
    """The oracle (single-threaded std::sort, untuned) on the host cores of
    this box, over the whole 1e8 input once; also confirms the GPU result.
    Beside it, the fast CPU baseline (per-thread std::nth_element over
    chunks, then a merge, on every host thread), labelled separately."""
    import oracle

    t0 = time.perf_counter()
    exp = oracle.topk_i32(x, K_TOP)
    t = time.perf_counter() - t0
    oracle.fast_topk_i32(x[:100000], K_TOP)  # build/load outside the timing
    ft = []
    for _ in range(3):
        t1 = time.perf_counter()
        fr, used = oracle.fast_topk_i32(x, K_TOP)
        ft.append(time.perf_counter() - t1)
    tf = statistics.median(ft)
    return {"value": round(x.size / t / 1e9, 5), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"the full {x.size}-element input, one call", "seconds": round(t, 3),
            "gpu_result_matches": bool(np.array_equal(exp, gpu_result)),
            "fast": {"kind": "per-thread std::nth_element over chunks + merge (not the oracle)",
                     "value": round(x.size / tf / 1e9, 4), "unit": UNIT, "seconds": round(tf, 4),
                     "cores": used, "hardware_concurrency": oracle.hardware_threads(), "cpu_model": cpu_model(),
                     "matches_oracle": bool(np.array_equal(fr, exp))}}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle, timed on bounded samples of the workload."""
    if rank != 0:
        return None
    import oracle

    n = synth.I32_WORKLOADS[WORKLOAD][1]
    # Calibrate the oracle's rate, then size a per-step sample so that the
    # whole run stays within about two minutes.
    probe = synth.i32_uniform(1_000_000, 2)
    t0 = time.perf_counter()
    oracle.topk_i32(probe, K_TOP)
    rate = probe.size / (time.perf_counter() - t0)
    budget = min(10.0, args.ref_budget_s / max(1, args.steps + args.warmup))
    m = int(min(n, max(10_000, rate * budget)))
    x = synth.i32_uniform(m, 2)  # the first m elements of the workload's input
    for _ in range(args.warmup):
        oracle.topk_i32(x, K_TOP)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.topk_i32(x, K_TOP)
    t = time.perf_counter() - t0
    value = m * args.steps / t / 1e9
    sample = f"first {m} elements of the workload's input per step"
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic: SplitMix64 uniform int32, seed 2",
        "config": {"workload": "int32 TopK, N=1e8 uniform full range (seed 2), k=20, output sorted descending",
                   "n": n, "k": K_TOP, "parallelism": "cpu oracle, rank 0"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


PROFILE_TARGETS = ("i32_1e8_k20", "i32_1e8_k100", "rows_tied", "rows_untied", "rows_untied_k129", "large_k1000_i32",
                   "large_k1000_f32", "sort_keys")


def run_profile_target(args):
    """A few calls of one workload and nothing else: the command that ncu
    captures take (`--profile NAME`); prints one short line."""
    import topk_selection_gb300 as tk

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    h = torch.cuda.current_stream(dev).cuda_stream
    name = args.profile
    if name.startswith("rows"):
        w = synth.ROWS_WORKLOAD
        xh = synth.f32_rows_tied(w["rows"], w["cols"], w["seed"], w["tie_frac"]) if name == "rows_tied" else \
            synth.f32_rows_normal(w["rows"], w["cols"], w["seed"])
        x = torch.from_numpy(xh).to(dev)
        rk = 129 if name == "rows_untied_k129" else w["k"]
        vals = torch.empty(w["rows"], rk, dtype=torch.float32, device=dev)
        idx = torch.empty(w["rows"], rk, dtype=torch.int32, device=dev)
        call = lambda: tk.topk_rows_f32_ptr(x.data_ptr(), w["rows"], w["cols"], rk, vals.data_ptr(),
                                            idx.data_ptr(), h)
    elif name == "sort_keys":
        x = torch.from_numpy(synth.i32_workload(WORKLOAD)).to(dev)
        ko = torch.empty_like(x)
        call = lambda: tk.sort_u32_ptr(x.data_ptr(), 0, x.numel(), ko.data_ptr(), 0, h)
    else:
        x = torch.from_numpy(synth.i32_workload(WORKLOAD)).to(dev)
        k = {"i32_1e8_k20": 20, "i32_1e8_k100": 100}.get(name, 1000)
        fn = tk.topk_f32_ptr if name.endswith("f32") else tk.topk_i32_ptr
        out = torch.empty(k, dtype=torch.int32, device=dev)
        call = lambda: fn(x.data_ptr(), x.numel(), k, out.data_ptr(), h)
    for _ in range(args.warmup + args.steps):
        rc = call()
        if rc != 0:
            raise tk.TopKError(rc, name)
    torch.cuda.synchronize()
    print(json.dumps({"profile": name, "calls": args.warmup + args.steps, "launches": tk.launch_count()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-cpu", action="store_true", help="leave out the CPU-baseline leg")
    ap.add_argument("--skip-rows", action="store_true", help="leave out the row-TopK, large-k, reduction, item and sort measurements")
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="--impl reference: seconds of oracle work for the whole run (sets the sample size)")
    ap.add_argument("--profile", choices=PROFILE_TARGETS, default=None,
                    help="run a few calls of one workload only (for ncu captures) and print a short line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile_target(args)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
