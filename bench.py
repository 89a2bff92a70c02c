#!/usr/bin/env python3
"""Benchmark of the batched verify-window MoE step on GB300.

A step is one window of the ``mid`` workload (d=2048, 128 experts top-8,
expert width 768, shared expert 768, 4-bit/32 blocks, fp32 router) at T=8
rows: router, grouping, gate/up, down and combine.  The headline is rows/s
with inputs resident in HBM and L2 flushed before every timed window; the
line also carries the T = 1, 2, 4, 8 sweep (rows/s, windows/s, algorithmic
GB/s), the gate/up kernel's roofline, an end-to-end figure through host
buffers, the GPU clocks seen, and the fp64 oracle timed on the host cores.

Multi-GPU: the step does not shard (one layer on one GPU); ``--gpus N`` under
torchrun runs N independent replicas and reports their summed rows over the
slowest rank's time.

``--impl reference`` times the fp64 oracle (the reference arm of this build)
on the host cores for the same metric: each step is one row of a T=8 window.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "rows/s per MoE window at T=8 (mid: d2048 E128 top8 F768 +shared768, 4-bit/32)"
UNIT = "rows/s"
N_WINDOWS = 64
SWEEP = (1, 2, 4, 8)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="mid")
    p.add_argument("--rows", type=int, default=8)
    p.add_argument("--sweep-steps", type=int, default=500)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-stack", action="store_true", help="skip the 48-layer stack measurement")
    p.add_argument("--no-head", action="store_true", help="skip the output-head measurement")
    p.add_argument("--no-workloads", action="store_true", help="skip the zipf and lowbit layer measurements")
    p.add_argument("--stack-steps", type=int, default=30)
    p.add_argument("--stack-layers", type=int, default=2, help="layers of the stack in --mode stack")
    p.add_argument("--mode", choices=("full", "windows", "stack", "head"), default="full",
                   help="windows / stack / head: only warmup + K launches of that kernel (a clean launch "
                        "sequence for ncu)")
    p.add_argument("--kv", action="store_true", help="--mode stack: attend over KV caches (positions ~1000)")
    return p.parse_args()


def bench_config(wl, T, world):
    """The workload keys of the JSON line, identical for both arms."""
    return {"workload": workload_desc(wl, T), "T": T, "windows": N_WINDOWS,
            "l2": "flushed before every timed window (memset of 2x L2 outside the events)",
            "parallelism": "replicas only" if world > 1 else "1 GPU"}


def workload_desc(wl, T):
    s = wl.moe
    return (f"{wl.name}: one MoE layer, d={s.hidden}, {s.n_experts} experts top-{s.top_k}, expert FFN {s.ffn}, "
            f"shared expert {s.shared_ffn}, {s.bits}-bit blocks of {s.block} (fp16 scale+min), fp32 router, "
            f"T={T} rows")


# ---------------------------------------------------------------------------------------------
# clocks


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.p = None
        time.sleep(0.3)

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) != 8:
                    continue
                try:
                    rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
                except ValueError:
                    continue
        os.unlink(self.f.name)
        if not rows:
            return None
        loaded = [r for r in rows if r[2] > 200.0] or rows
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in loaded:
            for n, v in zip(names, r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "samples_under_load": len(loaded),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------------------
# helpers


def flush_and_hold(flush):
    """Evict L2 (a memset of 2x its size), then keep the GPU busy for ~25 us
    with a spin kernel, so that the host enqueues the start event and the
    timed launch before the GPU reaches them (no host latency inside the
    device-timed region)."""
    import torch
    flush.zero_()
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(50000)


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy read+write)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback (6.8 TB/s, one earlier GB300 measurement)"


def kernel_source_hash():
    h = hashlib.sha1()
    for f in ("window.cu", "common.cuh", "frag.cuh"):
        with open(os.path.join(ROOT, "slot_decode_window_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source still matches it."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if line.startswith("traffic_bytes_per_launch:") or line.startswith("source_sha1:"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha1") != kernel_source_hash():
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def percentiles(vals):
    """(p10, median, p90) of a list, by linear interpolation between order statistics."""
    v = sorted(vals)

    def q(f):
        i = f * (len(v) - 1)
        lo = int(i)
        hi = min(lo + 1, len(v) - 1)
        return v[lo] + (v[hi] - v[lo]) * (i - lo)
    return q(0.1), q(0.5), q(0.9)


def oracle_subset(layer_np, xs):
    """The oracle's view of a layer holding only the routed experts the rows of
    the windows ``xs`` select (matrix stacks as {expert: array}), so that the
    child process that times the oracle receives a few hundred MB at most."""
    import oracle
    need = set()
    for x in xs:
        for t in range(x.shape[0]):
            need.update(int(e) for e in oracle.router(x[t], layer_np.router_w, layer_np.router_b,
                                                      layer_np.top_k, layer_np.renorm)[2])

    def sub(q):
        return oracle.OQMat({e: q.codes[e] for e in need}, {e: q.scale[e] for e in need},
                            {e: q.min[e] for e in need}, q.rows, q.cols, q.bits, q.block)
    import dataclasses
    return dataclasses.replace(layer_np, gate=sub(layer_np.gate), up=sub(layer_np.up), down=sub(layer_np.down))


def _time_oracle_child(job):
    """Runs in a spawned child: the fp64 oracle over whole windows; (seconds, rows)."""
    import oracle
    kind, payload, xs = job
    t0 = time.perf_counter()
    rows = 0
    for x in xs:
        if kind == "moe":
            oracle.moe_window(x, payload)
        else:  # one decoder layer, row by row
            dense, moe = payload
            for t in range(x.shape[0]):
                oracle.decoder_layer_row(x[t], dense, moe)
        rows += x.shape[0]
    return time.perf_counter() - t0, rows


def time_oracle(kind, payload, xs, threads):
    """The oracle timed in a fresh spawned process whose BLAS uses ``threads``
    threads (set through the environment before numpy loads in the child)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    names = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    old = {n: os.environ.get(n) for n in names}
    for n in names:
        os.environ[n] = str(threads)
    try:
        with cf.ProcessPoolExecutor(1, mp_context=mp.get_context("spawn")) as ex:
            sec, rows = ex.submit(_time_oracle_child, (kind, payload, xs)).result()
    finally:
        for n, v in old.items():
            if v is None:
                os.environ.pop(n, None)
            else:
                os.environ[n] = v
    return sec, rows


def cpu_baselines(jobs):
    """Each job (name, kind, payload, windows, T): the oracle with all host
    cores and with one, rows/s and windows/s."""
    out = {}
    cores = os.cpu_count() or 1
    for name, kind, payload, xs, T in jobs:
        entry = {"T": T, "windows": len(xs), "kind": "oracle"}
        for label, th in (("all_cores", cores), ("one_thread", 1)):
            sec, rows = time_oracle(kind, payload, xs, th)
            entry[label] = {"threads": th, "seconds": sec, "rows_per_s": rows / sec,
                            "windows_per_s": len(xs) / sec}
        out[name] = entry
    return out


# ---------------------------------------------------------------------------------------------
# reference arm: the oracle


def reduce_max_over_ranks(v: float, world: int, device) -> float:
    """The largest of v over all ranks (the slowest rank's time); v itself on one rank."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, seconds_max: float) -> float:
    """Units all ranks processed over the slowest rank's time (weak scaling)."""
    return units_per_rank * world / seconds_max


def run_reference(args, rank, world):
    if rank != 0:
        return
    import numpy as np
    from slot_decode_window_gb300 import workloads as wlm
    sys.path.insert(0, ROOT)
    from tests.helpers import omoe
    import oracle
    wl = wlm.WORKLOADS[args.workload]
    T = args.rows
    layer = wlm.make_moe_layer(wl.moe, seed=0, cfg_id=wl.cfg_id, device="cpu")
    ol = omoe(layer)
    xs = [wlm.make_window(wl, T, seed=0, window=w) for w in range(8)]
    rows = [(w, t) for w in range(len(xs)) for t in range(T)]
    for i in range(args.warmup):
        w, t = rows[i % len(rows)]
        oracle.moe_window(xs[w][t:t + 1], ol)
    t0 = time.perf_counter()
    for i in range(args.steps):
        w, t = rows[i % len(rows)]
        oracle.moe_window(xs[w][t:t + 1], ol)
    el = time.perf_counter() - t0
    value = args.steps / el
    cores = cpu_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(wl, T, world),
        "step": "one row of a T-row window, evaluated on its own by the fp64 oracle on the host cores (numpy BLAS)",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} rows cycled over 8 seeded windows of T={T}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
# our arm


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    from slot_decode_window_gb300 import binding, build, workloads as wlm

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0:
        build.build()
    if world > 1:
        torch.distributed.barrier()
        build.build()
    binding.load()

    wl = wlm.WORKLOADS[args.workload]
    spec = wl.moe
    d = spec.hidden
    layer = wlm.make_moe_layer(spec, seed=0, cfg_id=wl.cfg_id, device=str(dev))
    win = binding.Window(layer, max_rows=8)
    info = win.info()
    stream = torch.cuda.current_stream()

    if args.mode == "stack":
        # a short run of the decoder-layer stack kernel (for profilers): the
        # 48-layer stack's per-layer shapes, --stack-layers layers, T = --rows
        wls = wlm.WORKLOADS["stack48"]
        n = args.stack_layers
        moe = [wlm.make_moe_layer(wls.moe, seed=0, cfg_id=wls.cfg_id, layer=l, device=str(dev)) for l in range(n)]
        dense = [wlm.make_dense_layer(wls, seed=0, layer=l, device=str(dev)) for l in range(n)]
        stk = binding.Stack(wls, moe, dense, max_rows=8)
        T = args.rows
        xw = torch.from_numpy(np.stack([wlm.make_window(wls, T, seed=0, window=w) for w in range(4)])).to(dev)
        yw = torch.empty(T, wls.moe.hidden, device=dev)
        kw = {}
        if args.kv:
            shape = (n, 4, wls.kv_heads, 1024, wls.head_dim)
            kc = torch.randn(shape, device=dev).to(torch.float16)
            vc = torch.randn(shape, device=dev).to(torch.float16)
            stk.set_kv(kc, vc, 4, 1024)
            kw = dict(slot=torch.tensor([0, 0, 1, 1, 2, 2, 3, 3][:T], dtype=torch.int32, device=dev),
                      position=torch.tensor([1000, 1001] * 4, dtype=torch.int32, device=dev)[:T])
        for i in range(args.warmup + args.steps):
            stk.forward(xw[i % 4], yw, **kw)
        stk.sync()
        if rank == 0:
            print(json.dumps({"mode": "stack", "layers": n, "T": T, "windows": args.steps}), flush=True)
        stk.close()
        win.close()
        return

    if args.mode == "head":
        # the output head at the stack model's shape: warmup + K windows
        win.close()
        del layer
        torch.cuda.empty_cache()
        d, V, T = 2048, wlm.HEAD_VOCAB, args.rows
        W = wlm.make_head(V, d, 4, 32, seed=0, cfg_id=4, device=str(dev))
        head = binding.Head(W, max_rows=8)
        del W
        torch.cuda.empty_cache()
        xs = torch.randn(4, T, d, device=dev)
        pos = torch.arange(100, 100 + T, dtype=torch.int32, device=dev)
        seed = torch.full((T,), 12345, dtype=torch.int64, device=dev)
        temp = torch.tensor([0.0, 0.0, 0.7, 0.7, 0.0, 0.0, 1.0, 1.0][:T], device=dev)
        fed = torch.tensor([-1, 0] * 4, dtype=torch.int32, device=dev)[:T]
        for i in range(args.warmup + args.steps):
            head.forward(xs[i % 4], pos, seed, temp, fed)
        head.sync()
        if rank == 0:
            print(json.dumps({"mode": "head", "T": T, "windows": args.steps}), flush=True)
        head.close()
        return

    if args.mode == "windows":
        # the handle holds its own packed copy: free the unpacked tensors so a
        # profiler capture of a large layer keeps only that copy on the device
        del layer
        torch.cuda.empty_cache()
        T = args.rows
        xw = torch.from_numpy(np.stack([wlm.make_window(wl, T, seed=0, window=w) for w in range(N_WINDOWS)])).to(dev)
        yw = torch.empty(T, d, device=dev)
        for i in range(args.warmup + args.steps):
            win.forward(xw[i % N_WINDOWS], yw)
        win.sync()
        if rank == 0:
            print(json.dumps({"mode": "windows", "workload": args.workload, "T": T, "windows": args.steps}), flush=True)
        win.close()
        return

    Ts = sorted(set(SWEEP) | {args.rows})
    X = {T: torch.from_numpy(np.stack([wlm.make_window(wl, T, seed=0, window=1000 * T + w)
                                       for w in range(N_WINDOWS)])).to(dev) for T in Ts}
    Y = torch.empty(8, d, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    # distinct experts of every input window (from the library's own routing output)
    nd = {}
    for T in Ts:
        nd[T] = []
        for w in range(N_WINDOWS):
            _, rt = win.forward(X[T][w], Y[:T], routing=True)
            nd[T].append(int(rt["n_distinct"].item()))
    win.sync()

    eb, sb, rb = info.expert_bytes, info.shared_bytes, info.router_bytes

    def window_bytes(T, w):
        return nd[T][w] * eb + sb + rb + 2 * T * d * 4

    def timed(T, steps, warmup):
        for i in range(warmup):
            win.forward(X[T][i % N_WINDOWS], Y[:T])
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        t0 = time.perf_counter()
        for i in range(steps):
            flush_and_hold(flush)
            evs[i][0].record(stream)
            win.forward(X[T][i % N_WINDOWS], Y[:T])
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        if world > 1:
            torch.distributed.barrier()
        ms = [a.elapsed_time(b) for a, b in evs]
        nbytes = sum(window_bytes(T, i % N_WINDOWS) for i in range(steps))
        return ms, nbytes, wall

    def reduce_max(v):
        return reduce_max_over_ranks(v, world, dev)

    gpu_id = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    gpu_id = f"GPU-{gpu_id}" if gpu_id is not None and not str(gpu_id).startswith("GPU-") else str(gpu_id or local_rank)
    sampler = ClockSampler(gpu_id)

    # headline
    T = args.rows
    ms, nbytes, wall = timed(T, args.steps, max(3, args.warmup))
    total_s = reduce_max(sum(ms) / 1e3)
    value = whole_job_rate(args.steps * T, world, total_s)

    # sweep
    sweep = {}
    for Ts_ in SWEEP:
        m, b, _ = timed(Ts_, args.sweep_steps, 10)
        tot = sum(m) / 1e3
        q10, q50, q90 = percentiles(m)
        sweep[str(Ts_)] = {"rows_per_s": args.sweep_steps * Ts_ / tot, "windows_per_s": args.sweep_steps / tot,
                           "us_per_window_mean": 1e6 * tot / args.sweep_steps,
                           "us_per_window_p10": 1e3 * q10, "us_per_window_median": 1e3 * q50,
                           "us_per_window_p90": 1e3 * q90,
                           "algorithmic_GBps": b / tot / 1e9,
                           "mean_distinct_experts": sum(nd[Ts_]) / len(nd[Ts_])}

    # the same windows through the handle's CUDA-graph cache (fixed x/y buffers)
    xg = torch.empty(T, d, device=dev)
    yg = torch.empty(T, d, device=dev)
    for i in range(3):
        xg.copy_(X[T][i])
        win.forward_graph(xg, yg)
    g_ms = []
    for i in range(min(args.steps, 500)):
        xg.copy_(X[T][i % N_WINDOWS])
        flush_and_hold(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        win.forward_graph(xg, yg)
        b.record(stream)
        g_ms.append((a, b))
    torch.cuda.synchronize()
    g_ms = [a.elapsed_time(b) for a, b in g_ms]
    graph = {"T": T, "windows": len(g_ms), "us_per_window_median": 1e3 * statistics.median(g_ms),
             "rows_per_s": len(g_ms) * T / (sum(g_ms) / 1e3), "path": "strata_moe_window_forward_graph"}

    # window kernel roofline: events right around the kernel (profiling mode)
    win.set_profiling(True)
    prof_steps = min(args.steps, 400)
    k_ms = []
    wb = 0.0
    for i in range(prof_steps):
        flush_and_hold(flush)
        win.forward(X[T][i % N_WINDOWS], Y[:T])
        k_ms.append(win.timings())
        wb += window_bytes(T, i % N_WINDOWS)
    win.set_profiling(False)
    k_s = sum(k_ms) / 1e3
    peak, peak_src = measured_peak_hbm()
    achieved = wb / k_s / 1e9
    traffic = profiled_traffic("window_kernel", args.workload)
    roofline = {"kernel": "window_kernel<4> (router, grouping, gate/up, down, combine)", "bound": "hbm",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_src,
                "traffic": traffic, "algorithmic_bytes_per_launch": wb / prof_steps,
                "kernel_us_mean": 1e3 * statistics.mean(k_ms), "kernel_us_median": 1e3 * statistics.median(k_ms)}

    # the adaptive tier's bookkeeping attached (counters every window, a round every 4)
    tier = measure_tier(win, X[T], Y[:T], T, flush, min(args.steps, 300))

    # the output head of the stack model's shape (d 2048, V 151,936, 4-bit), T = 8
    head = None if args.no_head else measure_head(dev, flush, peak)

    # end to end through host buffers
    xh = torch.empty(N_WINDOWS, T, d, dtype=torch.float32).pin_memory()
    xh.copy_(X[T].cpu())
    yh = torch.empty(T, d, dtype=torch.float32).pin_memory()
    xd = torch.empty(T, d, device=dev)
    e2e_steps = min(args.steps, 1000)
    for i in range(5):
        xd.copy_(xh[i], non_blocking=True)
        win.forward(xd, Y[:T])
        yh.copy_(Y[:T], non_blocking=True)
    torch.cuda.synchronize()
    evs = []
    for i in range(e2e_steps):
        flush_and_hold(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        xd.copy_(xh[i % N_WINDOWS], non_blocking=True)
        win.forward(xd, Y[:T])
        yh.copy_(Y[:T], non_blocking=True)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    e2e_s = reduce_max(sum(a.elapsed_time(b) for a, b in evs) / 1e3)
    e2e = {"value": whole_job_rate(e2e_steps * T, world, e2e_s), "unit": UNIT, "h2d_bytes_per_step": T * d * 4,
           "d2h_bytes_per_step": T * d * 4}

    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    cpu_jobs = []
    if want_cpu:
        from tests.helpers import omoe
        xs = [X[T][w].cpu().numpy() for w in range(8)]
        cpu_jobs.append((args.workload, "moe", oracle_subset(omoe(layer), xs), xs, T))
    workloads = None
    if not args.no_workloads:
        workloads = {"zipf": measure_workload("zipf", (8,), dev, flush, stream, peak, cpu_jobs if want_cpu else None),
                     "lowbit": measure_workload("lowbit", (1, 2, 4, 8), dev, flush, stream, peak,
                                                cpu_jobs if want_cpu else None)}
    stack = None if args.no_stack else measure_stack(args, dev, flush, stream, peak, cpu_jobs if want_cpu else None)
    clocks = sampler.stop()
    # DRAM bytes per launch from the committed ncu summaries (null when the
    # kernel source changed since they were taken)
    if workloads:
        for wl_name, entry in workloads.items():
            if "8" in entry:
                entry["8"]["traffic"] = profiled_traffic("window_kernel_direct", wl_name)
    if stack:
        t2 = profiled_traffic("stack_kernel", "stack48_2layers")
        stack["traffic_per_layer"] = t2 / 2 if t2 is not None else None

    cpu = cpu_all = None
    if want_cpu:
        cpu_all = cpu_baselines(cpu_jobs)
        own = cpu_all[args.workload]
        cpu = {"value": own["all_cores"]["rows_per_s"], "unit": UNIT, "cores": own["all_cores"]["threads"],
               "kind": "oracle",
               "sample": f"{own['windows']} windows of T={T} of the bench's inputs, each window evaluated row by "
                         f"row by the fp64 oracle in a spawned process with {own['all_cores']['threads']} BLAS "
                         f"threads, {own['all_cores']['seconds']:.1f} s",
               "one_thread": own["one_thread"]}
    p10, p50, p90 = percentiles(ms)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": bench_config(wl, T, world),
            "arith": "codes -> exact fp16 integers; mma.sync f16 x (fp16 hi + lo activations), fp32 accumulate; "
                     "fp32 router, softmax, SwiGLU, combine",
            "roofline": roofline, "sweep": sweep, "graph": graph, "tier": tier, "head": head, "workloads": workloads,
            "stack48": stack, "e2e": e2e,
            "clocks": clocks,
            "cpu_baseline": cpu, "cpu_baselines": cpu_all,
            "gpu_launches": args.steps,
            "window_us": {"mean": 1e3 * statistics.mean(ms), "p10": 1e3 * p10, "median": 1e3 * p50, "p90": 1e3 * p90},
            "rows_per_s_at_median": T / (p50 / 1e3), "wall_s_timed_region": wall,
            "handle": {"n_sm": info.n_sm, "stages": info.stages, "stage_bytes": info.stage_bytes,
                       "smem_bytes": info.smem_bytes},
        }
        print(json.dumps(line), flush=True)
    win.close()


def measure_head(dev, flush, peak, steps=200):
    """The output head at the 48-layer stack's model shape (d 2048, V 151,936,
    4-bit/32): a T = 8 window of 4 slots x (token, proposal), half greedy and
    half sampled rows; kernel time from profiling-mode events, L2 flushed
    before each window.  Algorithmic bytes: the head's block bytes, the rows
    of x, and the logits written once and read by the draw."""
    import numpy as np
    import torch
    from slot_decode_window_gb300 import binding, workloads as wlm
    d, V, T = 2048, wlm.HEAD_VOCAB, 8
    W = wlm.make_head(V, d, 4, 32, seed=0, cfg_id=4, device=str(dev))
    head = binding.Head(W, max_rows=8)
    del W
    torch.cuda.empty_cache()
    hb = head.head_bytes()
    xs = torch.from_numpy(np.random.default_rng(0).standard_normal((16, T, d)).astype(np.float32)).to(dev)
    pos = torch.arange(100, 100 + T, dtype=torch.int32, device=dev)
    seed = torch.full((T,), 12345, dtype=torch.int64, device=dev)
    temp = torch.tensor([0.0, 0.0, 0.7, 0.7, 0.0, 0.0, 1.0, 1.0], device=dev)
    fed = torch.tensor([-1, 0, -1, 0, -1, 0, -1, 0], dtype=torch.int32, device=dev)
    for i in range(5):
        head.forward(xs[i % 16], pos, seed, temp, fed)
    head.set_profiling(True)
    ms = []
    for i in range(steps):
        flush_and_hold(flush)
        head.forward(xs[i % 16], pos, seed, temp, fed)
        ms.append(head.timings())
    head.set_profiling(False)
    head.sync()
    head.close()
    nbytes = hb + T * d * 4 + 2 * T * V * 4
    mean_s = statistics.mean(ms) / 1e3
    q10, q50, q90 = percentiles(ms)
    return {"workload": "output head d 2048, V 151,936, 4-bit/32, T = 8 (4 slots x (token, proposal)), "
                        "greedy and sampled rows, proposal check",
            "kernel": "head_kernel<4> (RMSNorm, head GEMV, draw, proposal check; one cooperative launch)",
            "us_per_window_mean": 1e6 * mean_s, "us_per_window_p10": 1e3 * q10, "us_per_window_median": 1e3 * q50,
            "us_per_window_p90": 1e3 * q90, "algorithmic_bytes": nbytes, "achieved_GBps": nbytes / mean_s / 1e9,
            "frac_of_measured_hbm": nbytes / mean_s / 1e9 / peak, "rows_per_s": T / mean_s,
            "traffic": profiled_traffic("head_kernel", "d2048_v151936")}


def measure_tier(win, X, Y, T, flush, steps):
    """Window kernel time with an adaptive tier attached (capacity E/2, a round
    every 4 windows, up to 8 swaps, decay 0.5, min gain 1.5) against the same
    windows without one, profiling-mode events around the launch."""
    from slot_decode_window_gb300 import binding as B
    E = win.spec.n_experts
    st, tier = B.strata_tier_create(B.strata_tier_desc(E, max(1, E // 2), 4, 8, 0.5, 1.5))
    B.check(st, "strata_tier_create")
    out = {}
    try:
        for label, t in (("without", None), ("with", tier)):
            B.check(B.strata_window_set_tier(win.handle, t), "strata_window_set_tier")
            win.set_profiling(True)
            ms = []
            for i in range(steps):
                flush_and_hold(flush)
                win.forward(X[i % N_WINDOWS], Y)
                ms.append(win.timings())
            win.set_profiling(False)
            out[f"kernel_us_mean_{label}_tier"] = 1e3 * statistics.mean(ms)
        B.check(B.strata_window_set_tier(win.handle, None), "strata_window_set_tier")
        st, state = B.strata_tier_read(tier, E)
        B.check(st, "strata_tier_read")
        out.update(T=T, windows=steps, rounds=int(state["rounds"]), last_round_swaps=int(state["n_swaps"]),
                   overhead_us=out["kernel_us_mean_with_tier"] - out["kernel_us_mean_without_tier"],
                   tier="capacity E/2, a round every 4 windows, up to 8 swaps, decay 0.5, min gain 1.5")
    finally:
        B.strata_window_set_tier(win.handle, None)
        B.strata_tier_destroy(tier)
    return out


def measure_workload(name, Ts, dev, flush, stream, peak, cpu_jobs=None, steps=300):
    """Another layer shape of the pages' workloads at the given row counts:
    mean kernel time per window (profiling-mode events around the launch, L2
    flushed before each window) over its algorithmic bytes.  With cpu_jobs, a
    job timing the oracle on three T = max(Ts) windows of this layer is added."""
    import numpy as np
    import torch
    from slot_decode_window_gb300 import binding, workloads as wlm
    wl = wlm.WORKLOADS[name]
    layer = wlm.make_moe_layer(wl.moe, seed=0, cfg_id=wl.cfg_id, device=str(dev))
    win = binding.Window(layer, max_rows=8)
    if cpu_jobs is not None:
        from tests.helpers import omoe_lazy
        Tc = max(Ts)
        xs = [wlm.make_window(wl, Tc, seed=0, window=2000 * Tc + w) for w in range(3)]
        cpu_jobs.append((name, "moe", oracle_subset(omoe_lazy(layer), xs), xs, Tc))
    del layer
    torch.cuda.empty_cache()
    info = win.info()
    d = wl.moe.hidden
    out = {"workload": workload_desc(wl, "|".join(str(t) for t in Ts))}
    for T in Ts:
        X = torch.from_numpy(np.stack([wlm.make_window(wl, T, seed=0, window=2000 * T + w) for w in range(16)])).to(dev)
        Y = torch.empty(T, d, device=dev)
        nd = []
        for w in range(16):
            _, rt = win.forward(X[w], Y, routing=True)
            nd.append(int(rt["n_distinct"].item()))
        win.sync()
        wb = [n * info.expert_bytes + info.shared_bytes + info.router_bytes + 2 * T * d * 4 for n in nd]
        for i in range(5):
            win.forward(X[i % 16], Y)
        win.set_profiling(True)
        ms, nbytes = [], 0.0
        for i in range(steps):
            flush_and_hold(flush)
            win.forward(X[i % 16], Y)
            ms.append(win.timings())
            nbytes += wb[i % 16]
        win.set_profiling(False)
        win.sync()
        tot = sum(ms) / 1e3
        achieved = nbytes / tot / 1e9
        q10, q50, q90 = percentiles(ms)
        out[str(T)] = {"us_per_window_mean": 1e6 * tot / steps, "us_per_window_p10": 1e3 * q10,
                       "us_per_window_median": 1e3 * q50, "us_per_window_p90": 1e3 * q90,
                       "rows_per_s": steps * T / tot,
                       "windows_per_s": steps / tot, "algorithmic_MB_per_window": nbytes / steps / 1e6,
                       "mean_distinct_experts": sum(nd) / len(nd), "achieved_GBps": achieved,
                       "frac_of_measured_hbm": achieved / peak}
    win.close()
    return out


def measure_stack(args, dev, flush, stream, peak, cpu_jobs=None):
    """The 48-layer decoder stack (dense 4-bit q/k/v/o + the mid MoE per layer),
    T = 8, one launch per window, L2 flushed before each window.  With
    cpu_jobs, a job timing the oracle on one window through one layer (the
    stack's per-layer cost; a window through all layers is 48 of these) is added."""
    import numpy as np
    import torch
    from slot_decode_window_gb300 import binding, workloads as wlm
    wl = wlm.WORKLOADS["stack48"]
    moe = [wlm.make_moe_layer(wl.moe, seed=0, cfg_id=wl.cfg_id, layer=l, device=str(dev)) for l in range(wl.n_layers)]
    dense = [wlm.make_dense_layer(wl, seed=0, layer=l, device=str(dev)) for l in range(wl.n_layers)]
    if cpu_jobs is not None:
        from tests.helpers import odense, omoe
        cpu_jobs.append(("stack48_one_layer", "layer", (odense(dense[0], wl), omoe(moe[0])),
                         [wlm.make_window(wl, 8, seed=0, window=0)], 8))
    stk = binding.Stack(wl, moe, dense, max_rows=8)
    del moe, dense
    torch.cuda.empty_cache()
    info = stk.info()
    T, nw = 8, 8
    X = torch.from_numpy(np.stack([wlm.make_window(wl, T, seed=0, window=w) for w in range(nw)])).to(dev)
    Y = torch.empty(T, wl.moe.hidden, device=dev)
    per_window = []
    for w in range(nw):
        _, res = stk.forward(X[w], Y, outputs=True)
        ndl = res["n_distinct"].cpu().numpy()
        per_window.append(float(ndl.sum() * info.expert_bytes
                                + wl.n_layers * (info.shared_bytes + info.router_bytes + info.dense_bytes)
                                + 2 * T * wl.moe.hidden * 4))
    stk.sync()
    steps, warm = args.stack_steps, 3
    for i in range(warm):
        stk.forward(X[i % nw], Y)
    stk.set_profiling(True)
    ms = []
    nbytes = 0.0
    for i in range(steps):
        flush_and_hold(flush)
        stk.forward(X[i % nw], Y)
        ms.append(stk.timings())
        nbytes += per_window[i % nw]
    stk.set_profiling(False)
    stk.sync()
    tot = sum(ms) / 1e3
    achieved = nbytes / tot / 1e9
    out = {"workload": "48 layers x (RMSNorm, dense 4-bit q/k/v/o 2048->4096/512/512, o 4096->2048, "
                       "MoE d2048 E128 k8 F768 + shared 768), T=8",
           "windows": steps, "warmup": warm, "ms_per_window_median": statistics.median(ms),
           "rows_per_s": steps * T / tot, "algorithmic_bytes_per_window": nbytes / steps,
           "achieved_GBps": achieved, "peak_GBps": peak, "frac": achieved / peak,
           "kernel": "stack_kernel<4> (one cooperative launch per window)", "gpu_launches_per_window": 1}

    # the same stack attending over each slot's KV cache: 4 slots x (token,
    # proposal) at positions 1000 and 1001 over 1000 positions of history
    n_slots, max_ctx, hist = 4, 1024, 1000
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    shape = (wl.n_layers, n_slots, wl.kv_heads, max_ctx, wl.head_dim)
    kc = torch.randn(shape, generator=g, device=dev).to(torch.float16)
    vc = torch.randn(shape, generator=g, device=dev).to(torch.float16)
    stk.set_kv(kc, vc, n_slots, max_ctx)
    slot = torch.tensor([0, 0, 1, 1, 2, 2, 3, 3], dtype=torch.int32, device=dev)
    pos = torch.tensor([hist, hist + 1] * 4, dtype=torch.int32, device=dev)
    kv_bytes = wl.n_layers * n_slots * 2 * wl.kv_heads * (hist + 2) * wl.head_dim * 2
    for i in range(warm):
        stk.forward(X[i % nw], Y, slot=slot, position=pos)
    stk.set_profiling(True)
    ms2, nb2 = [], 0.0
    for i in range(steps):
        flush_and_hold(flush)
        stk.forward(X[i % nw], Y, slot=slot, position=pos)
        ms2.append(stk.timings())
        nb2 += per_window[i % nw] + kv_bytes
    stk.set_profiling(False)
    stk.sync()
    tot2 = sum(ms2) / 1e3
    out["with_kv_cache"] = {
        "workload": "the same 48 layers attending over fp16 KV caches: 4 slots x (token, proposal) rows at "
                    "positions 1000 and 1001, 1000 positions of history per slot",
        "ms_per_window_median": statistics.median(ms2), "rows_per_s": steps * T / tot2,
        "kv_bytes_per_window": kv_bytes, "algorithmic_bytes_per_window": nb2 / steps,
        "achieved_GBps": nb2 / tot2 / 1e9, "frac": nb2 / tot2 / 1e9 / peak}
    stk.close()
    return out


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)  # rank 0 only; the other ranks exit at once
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
