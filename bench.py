"""Benchmark: CSR SpMV y = alpha*A*x + beta*y on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--all] [--impl reference]

One step is one product through the C ABI with every input resident in HBM
(plan built beforehand, its time reported as plan_ms).  W untimed steps,
then exactly K timed steps between a barrier and a device synchronisation,
each bracketed by CUDA events on the launching stream.  Prints one JSON line
(rank 0).  The default workload is the 3-D 27-point stencil on a 128^3 grid
(fp32, 55.7M nonzeros, 479.5 MB of compulsory traffic -- larger than L2, so
no flush between steps; x stays L2-resident as in an iterative solver).

--gpus N > 1 (under torchrun): N independent replicas, one per GPU, each on
the full workload; the product has no exchange step on one matrix per GPU
(weak scaling, value = all ranks' flops / max time over ranks).

--impl reference: the CPU oracle (single-threaded, long double) timed on a
bounded sample of the same workload, as the reference arm.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import platform
import shutil
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "SpMV GFLOP/s and achieved HBM GB/s (% of roofline) per matrix, 1 GB300"
DEFAULT_WORKLOAD = "stencil27_128"
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def compulsory_bytes(A, beta: float | None = None) -> int:
    """B_c = nnz*(4+s) + (m+1)*4 + n*s + 2*m*s: every column index and value
    once, row_ptr once, x once, y read and written once (the bytes-per-nonzero
    model of the Row-grouped CSR page, section 3, extended by row_ptr, x and
    y).  This is the roofline's byte count.  With beta given, the count the
    product actually needs: y is only written when beta == 0 (BLAS
    convention), so m*s fewer bytes."""
    s = A.vals.dtype.itemsize
    y_bytes = 2 * A.m * s if beta is None or beta != 0 else A.m * s
    return A.nnz * (4 + s) + (A.m + 1) * 4 + A.n * s + y_bytes


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources each product kernel is built from
KERNEL_SOURCES = {
    "merge_path": ["merge_path.cu", "tma.cuh", "internal.cuh"],
    "rgcsr": ["rgcsr.cu", "long_rows.cu", "tma.cuh", "internal.cuh"],
    "long_rows": ["long_rows.cu", "row_kernels.cu", "internal.cuh"],
    "thread_row": ["row_kernels.cu", "internal.cuh"],
}


def kernel_source_hash(kernel: str | None = None) -> str:
    """Hash of one kernel's sources (all of csrc/ when kernel is None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "load_balanced_csr_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) if kernel else None
    if names is None:
        names = [n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh"))]
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None, None
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None, None
    return e.get("dram_bytes_per_launch"), e.get("note")


def roofline(bc: int, bc_beta: int, mean_us: float, workload: str, kernel: str) -> dict:
    """The product's roofline entry: B_c (y read and written) over the mean
    CUDA-event time of one product, against the measured copy bandwidth and
    the 8 TB/s spec; frac_beta_aware uses the bytes the product needs (no y
    read when beta == 0)."""
    peak, peak_kind = measured_peak()
    achieved = bc / (mean_us * 1e-6) / 1e9
    achieved_b = bc_beta / (mean_us * 1e-6) / 1e9
    traffic, traffic_note = recorded_traffic(workload, kernel)
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} copy bandwidth",
            "frac_of_spec_8tbs": round(achieved / SPEC_HBM_GBS, 4),
            "frac_beta_aware": round(achieved_b / peak, 4), "traffic": traffic, "kernel": kernel,
            "algorithmic_bytes_per_launch": int(bc), "beta_aware_bytes_per_launch": int(bc_beta)}
    if traffic_note:
        roof["traffic_note"] = traffic_note
    return roof


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int):
        self.proc = None
        self.err = None
        exe = shutil.which("nvidia-smi")
        if not exe:
            self.err = "nvidia-smi not found"
            return
        sel = self._select(device_index)
        self.path = os.path.join(tempfile.gettempdir(), f"spmv_clocks_{os.getpid()}.csv")
        self.fh = open(self.path, "w")
        self.proc = subprocess.Popen([exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                      "-lms", "50", "-i", sel], stdout=self.fh, stderr=subprocess.DEVNULL)

    @staticmethod
    def _select(device_index: int) -> str:
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            return vis.split(",")[device_index] if vis else str(device_index)

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"unavailable": self.err}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.03 <= r[0] <= t1 + 0.03]
        window = "timed region"
        if not inside:
            inside, window = rows, "sampler run (timed region shorter than one sample)"
        if not inside:
            return {"unavailable": "no samples"}
        reasons = sorted({self.NAMES[i] for r in inside for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------------ GPU arm


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(v: float, world: int, device=None) -> float:
    """The largest v over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gflops(nnz: int, world: int, ms_per_step: float, k: int = 1) -> float:
    """Whole-job throughput: every rank runs one product of 2*nnz*k flops per
    step (replicas), over the slowest rank's time per step."""
    return 2.0 * nnz * k * world / (ms_per_step * 1e-3) / 1e9


def run_gpu(args, workload_name: str) -> dict | None:
    import torch
    import torch.distributed as dist

    import load_balanced_csr_gb300 as lb

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    W = synth.workload(workload_name)
    A = W.A
    vt = torch.float64 if A.dtype == "f64" else torch.float32
    rp = torch.from_numpy(A.row_ptr).to(dev)
    col = torch.from_numpy(A.col_idx).to(dev)
    val = torch.from_numpy(A.vals).to(dev)
    x = torch.from_numpy(W.x).to(dev)
    y0 = torch.from_numpy(W.y0).to(dev) if W.y0 is not None else None
    y = y0.clone() if y0 is not None else torch.zeros(A.m, dtype=vt, device=dev)
    stream = torch.cuda.current_stream(dev)

    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    plan = lb.Plan(rp, col, val, A.n, kernel=args.kernel, items_per_thread=args.ipt, rgcsr_group=args.group,
                   long_row_min=args.long_min, with_transpose=args.transposed)
    torch.cuda.synchronize(dev)
    plan_ms = (time.perf_counter() - t) * 1e3
    info = plan.info()
    run = plan.execute_transposed if args.transposed else plan  # the workloads are square: x, y fit both ways
    if args.transposed:
        info["kernel_name"] = lb.KERNEL_NAMES.get(info["transposed_kernel"], "?") + " (A^T)"
        info["launches_per_execute"] = info["transposed_launches"]

    for _ in range(args.warmup):
        run(x, y, W.alpha, W.beta, stream)
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.15 if sampler else 0)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    start_all = torch.cuda.Event(enable_timing=True)
    end_all = torch.cuda.Event(enable_timing=True)
    start_all.record(stream)
    for k in range(K):
        ev[k][0].record(stream)
        run(x, y, W.alpha, W.beta, stream)
        ev[k][1].record(stream)
    end_all.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    t1 = time.time()
    clocks = sampler.stop(t0, t1) if sampler else None

    total_ms = max_over_ranks(start_all.elapsed_time(end_all), world, dev)
    per = np.array([a.elapsed_time(b) for a, b in ev]) * 1e3  # us

    # end to end through the public API: pinned host x in (and y when beta !=
    # 0), host y out, every step.  The product goes through spmv_execute_host,
    # which queues the copies and the product itself; the transposed product
    # has no host entry point, so its copies are queued by torch around
    # spmv_execute_transposed.  With beta != 0 each step reads the previous
    # step's y: the same bytes and work as a product from fixed inputs.
    e2e = None
    if True:
        x_h = torch.from_numpy(W.x).pin_memory()
        y_h = torch.from_numpy(W.y0.copy()).pin_memory() if W.y0 is not None else torch.empty(A.m, dtype=vt).pin_memory()
        if args.transposed:
            def e2e_step():
                x.copy_(x_h, non_blocking=True)
                if W.y0 is not None:
                    y.copy_(y_h, non_blocking=True)
                run(x, y, W.alpha, W.beta, stream)
                y_h.copy_(y, non_blocking=True)
            e2e_api = "torch copies around spmv_execute_transposed"
        else:
            def e2e_step():
                plan.execute_host(x_h, y_h, x, y, W.alpha, W.beta, stream)
            e2e_api = "spmv_execute_host (the library queues the copies and the product)"
        ke = max(3, min(K, args.e2e_steps))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        s_e, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_e.record(stream)
        for _ in range(ke):
            e2e_step()
        e_e.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(s_e.elapsed_time(e_e) / ke, world, dev)
        s = A.vals.dtype.itemsize
        h2d = A.n * s + (A.m * s if W.y0 is not None else 0)
        e2e = {"value": round(job_gflops(A.nnz, world, e2e_ms), 3), "unit": "GFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(A.m * s), "ms_per_step": round(e2e_ms, 4),
               "steps": ke, "api": e2e_api}
    plan.close()
    if rank != 0:
        return None

    ms_step = total_ms / K
    bc = compulsory_bytes(A)
    bc_beta = compulsory_bytes(A, W.beta)
    gflops = job_gflops(A.nnz, world, ms_step)
    mean_us = float(per.mean())
    roof = roofline(bc, bc_beta, mean_us, workload_name, info["kernel_name"])
    out = {
        "metric": METRIC, "value": round(gflops, 3), "unit": "GFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": A.dtype, "data": "synthetic",
        "config": {"workload": workload_name, "description": W.description, "m": A.m, "n": A.n, "nnz": A.nnz,
                   "alpha": W.alpha, "beta": W.beta, "kernel": info["kernel_name"],
                   "items_per_tile": info["items_per_tile"], "num_tiles": info["num_tiles"],
                   "l2": "inputs larger than L2, no flush (x stays L2-resident across steps)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "gbs_effective": roof["achieved"],
        "median_us": round(float(np.median(per)), 3), "p10_us": round(float(np.percentile(per, 10)), 3),
        "p90_us": round(float(np.percentile(per, 90)), 3), "compulsory_bytes": int(bc),
        "plan_ms": round(plan_ms, 3), "roofline": roof,
        "gpu_launches": int(K * info["launches_per_execute"]),
        "e2e": e2e, "clocks": clocks,
    }
    return out


# ------------------------------------------------------------------ CPU oracle arm


def oracle_sample(W, budget_s: float):
    """Time the oracle on a leading block of rows sized to ~budget_s seconds."""
    import oracle
    A = W.A
    lens = np.diff(A.row_ptr.astype(np.int64))
    cum = np.cumsum(lens)

    def rows_for(nnz_target):
        r = int(np.searchsorted(cum, nnz_target)) + 1
        return max(1, min(A.m, r))

    def run(r):
        rows = np.arange(r, dtype=np.int32)
        t = time.perf_counter()
        oracle.spmv(A.row_ptr, A.col_idx, A.vals, W.x, W.alpha, W.beta, W.y0, rows=rows)
        return time.perf_counter() - t

    r = rows_for(200_000)
    t = run(r)
    nnz_r = int(A.row_ptr[r])
    rate = max(nnz_r, 1) / max(t, 1e-6)
    r = rows_for(rate * budget_s)
    return r, int(A.row_ptr[r])


def copy_bandwidth(dev) -> float:
    """Device copy bandwidth measured in this run: b.copy_(a) over 1 GiB of
    bf16 (read + write bytes), best of 10, CUDA events -- the method of the
    measured peak, repeated on this machine."""
    import torch
    a = torch.empty(1 << 29, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    a.fill_(1.0)
    best = float("inf")
    for _ in range(12):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize(dev)
        best = min(best, e0.elapsed_time(e1))
    del a, b
    torch.cuda.empty_cache()
    return 2 * (1 << 30) / (best * 1e-3) / 1e9


def per_config_entry(name: str, dev, warmup: int, min_runs: int, min_seconds: float, cpu_budget: float,
                     copy_gbs: float | None) -> dict:
    """One workload with the plan's own kernel choice: median time per product
    over at least min_runs runs (and at least min_seconds of them, so that the
    clock sampler sees the timed region), one CUDA event pair per run, inputs
    larger than L2 and no flush between runs; GFLOP/s = 2*nnz/t, GB/s =
    B_c/t and the roofline fractions with t the median; the oracle on a
    bounded sample of rows on one host core."""
    import torch
    import load_balanced_csr_gb300 as lb
    W = synth.workload(name)
    A = W.A
    vt = torch.float64 if A.dtype == "f64" else torch.float32
    rp = torch.from_numpy(A.row_ptr).to(dev)
    col = torch.from_numpy(A.col_idx).to(dev)
    val = torch.from_numpy(A.vals).to(dev)
    x = torch.from_numpy(W.x).to(dev)
    y = torch.from_numpy(W.y0).to(dev) if W.y0 is not None else torch.zeros(A.m, dtype=vt, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    plan = lb.Plan(rp, col, val, A.n)
    torch.cuda.synchronize(dev)
    plan_ms = (time.perf_counter() - t) * 1e3
    info = plan.info()
    for _ in range(max(warmup, 10)):
        plan(x, y, W.alpha, W.beta, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(5):
        plan(x, y, W.alpha, W.beta, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    est_us = e0.elapsed_time(e1) * 1e3 / 5
    runs = int(min(5000, max(min_runs, min_seconds / max(est_us * 1e-6, 1e-7))))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
    sampler = ClockSampler(dev.index or 0)
    time.sleep(0.15)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for a, b in ev:
        a.record(stream)
        plan(x, y, W.alpha, W.beta, stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop(t0, time.time())
    status = plan.device_status()
    plan.close()
    per = np.array([a.elapsed_time(b) for a, b in ev]) * 1e3
    med = float(np.median(per))
    bc, bc_beta = compulsory_bytes(A), compulsory_bytes(A, W.beta)
    peak, peak_kind = measured_peak()
    gbs = bc / (med * 1e-6) / 1e9
    traffic = recorded_traffic(name, info["kernel_name"])[0]
    entry = {
        "workload": name, "description": W.description, "kernel": info["kernel_name"], "dtype": A.dtype,
        "m": A.m, "n": A.n, "nnz": A.nnz, "alpha": W.alpha, "beta": W.beta, "runs": runs, "warmup": max(warmup, 10),
        "median_us": round(med, 3), "mean_us": round(float(per.mean()), 3),
        "p10_us": round(float(np.percentile(per, 10)), 3), "p90_us": round(float(np.percentile(per, 90)), 3),
        "gflops": round(2.0 * A.nnz / (med * 1e-6) / 1e9, 2), "gbs_effective": round(gbs, 1),
        "roofline": {"bound": "hbm", "time": "median", "bytes": int(bc), "beta_aware_bytes": int(bc_beta),
                     "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "peak_source": f"{peak_kind} copy bandwidth",
                     "frac": round(gbs / peak, 4),
                     "frac_beta_aware": round(bc_beta / (med * 1e-6) / 1e9 / peak, 4),
                     "frac_of_spec_8tbs": round(gbs / SPEC_HBM_GBS, 4),
                     "frac_of_copy_this_run": round(gbs / copy_gbs, 4) if copy_gbs else None,
                     "meets_70pct": bool(gbs / peak >= 0.70)},
        # DRAM bytes per launch from the committed ncu capture of this kernel on
        # this workload, when it was taken on the current sources (else null),
        # and their ratio to the bytes the product needs
        "traffic": traffic,
        "traffic_over_needed": round(traffic / bc_beta, 3) if traffic else None,
        "plan_ms": round(plan_ms, 3), "launches_per_execute": info["launches_per_execute"],
        "items_per_tile": info["items_per_tile"], "num_tiles": info["num_tiles"],
        "device_status": status, "clocks": clocks,
        "l2": "inputs larger than L2 (laplace2d_64 excepted), no flush between runs",
    }
    del rp, col, val, x, y
    torch.cuda.empty_cache()
    entry["cpu_baseline"] = cpu_baseline_leg(name, cpu_budget) if cpu_budget > 0 else None
    return entry


def run_per_config(args) -> dict:
    """Every workload on one GPU: each one's median time per product,
    GFLOP/s, GB/s and roofline fractions, with the oracle beside it."""
    import torch
    _, _, local = dist_env()
    dev = torch.device("cuda", local)
    copy_gbs = copy_bandwidth(dev)
    entries = [per_config_entry(name, dev, args.warmup, 100, 0.3, args.per_config_cpu_budget, copy_gbs)
               for name in synth.WORKLOADS]
    return {"copy_gbs_this_run": round(copy_gbs, 1), "configs": entries}


def run_reference(args, workload_name: str) -> dict | None:
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    W = synth.workload(workload_name)
    A = W.A
    per_step = max(0.05, min(1.0, 150.0 / max(1, args.steps + args.warmup)))
    r, nnz_s = oracle_sample(W, per_step)
    rows = np.arange(r, dtype=np.int32)
    for _ in range(args.warmup):
        oracle.spmv(A.row_ptr, A.col_idx, A.vals, W.x, W.alpha, W.beta, W.y0, rows=rows)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.spmv(A.row_ptr, A.col_idx, A.vals, W.x, W.alpha, W.beta, W.y0, rows=rows)
        times.append(time.perf_counter() - t)
    tot = float(np.sum(times))
    gflops = 2.0 * nnz_s * args.steps / tot / 1e9
    sample = f"rows [0, {r}) of {A.m} ({nnz_s} of {A.nnz} nonzeros) per step"
    return {
        "metric": METRIC, "value": round(gflops, 4), "unit": "GFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": A.dtype, "data": "synthetic", "impl": "reference",
        "config": {"workload": workload_name, "description": W.description, "m": A.m, "n": A.n, "nnz": A.nnz,
                   "alpha": W.alpha, "beta": W.beta},
        "cpu_baseline": {"value": round(gflops, 4), "unit": "GFLOP/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "cpu": cpu_model()},
        "e2e": {"value": round(gflops, 4), "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                low = line.lower()
                if low.startswith("model name") or low.startswith("cpu part") or low.startswith("hardware"):
                    return f"{platform.machine()} {line.split(':', 1)[1].strip()} ({os.cpu_count()} cores)"
    except Exception:
        pass
    return f"{platform.machine()} ({os.cpu_count()} cores)"


def cpu_baseline_leg(workload_name: str, budget_s: float) -> dict:
    import oracle
    W = synth.workload(workload_name)
    A = W.A
    r, nnz_s = oracle_sample(W, budget_s / 3)
    rows = np.arange(r, dtype=np.int32)
    ts = []
    for _ in range(3):
        t = time.perf_counter()
        oracle.spmv(A.row_ptr, A.col_idx, A.vals, W.x, W.alpha, W.beta, W.y0, rows=rows)
        ts.append(time.perf_counter() - t)
    t = float(np.median(ts))
    return {"value": round(2.0 * nnz_s / t / 1e9, 4), "unit": "GFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"rows [0, {r}) of {A.m} ({nnz_s} of {A.nnz} nonzeros), median of 3, long double",
            "cpu": cpu_model()}


def spmm_path_of(info: dict, k: int, s: int, row_ptr):
    """(name, launches) of the SpMM path spmv_execute_multi takes for this
    plan with contiguous, 16-byte aligned X and Y of k columns (the choice
    made in the library's spmv_execute_multi, restated for the report)."""
    kmax = 16 if s == 8 else 32
    w = 16 // s
    if info["kernel_name"] in ("rgcsr", "rgcsr_sorted") and info["rgcsr_group"] == 32 and \
            info["num_long_rows"] * 4096 <= info["m"]:
        if info["num_long_rows"] == 0:
            return "Row-grouped SpMM (thread per row; lanes share X rows from 4 lanes per row)", -(-k // kmax)
        return ("Row-grouped SpMM + a warp per 4096-nonzero segment of the long rows",
                -(-k // kmax) + -(-k // 32))
    n_long = int((np.diff(row_ptr) >= 65).sum())
    if (n_long == 0 or (n_long * 4096 <= info["m"] and k <= 2 * kmax)) and k % w == 0:
        slices, rest = 0, k
        while rest > 0:
            kc = kmax
            while kc > rest:
                kc //= 2
            rest -= kc
            slices += 1
        if n_long == 0:
            return "short-row SpMM from CSR (warp per 32 rows, lanes share X rows)", slices
        return ("CSR SpMM: warp per 32 short rows + warp per 4096-nonzero segment of the rows of 65 or more",
                2 * slices)
    return "merge-path SpMM (runs of warp tiles, lanes over columns)", -(-k // 128)


def run_spmm(args, workload_name: str) -> dict | None:
    """Y = alpha*A*X + beta*Y with k = args.rhs right-hand sides (row-major,
    seeded X) on the workload's matrix: GFLOP/s = 2*nnz*k/t and the
    algorithmic bytes nnz*(4+s) + (m+1)*4 + n*k*s + m*k*s*(1 + [beta != 0])."""
    import torch
    import load_balanced_csr_gb300 as lb

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    W = synth.workload(workload_name)
    A = W.A
    k = args.rhs
    vt = torch.float64 if A.dtype == "f64" else torch.float32
    s = A.vals.dtype.itemsize
    rp = torch.from_numpy(A.row_ptr).to(dev)
    col = torch.from_numpy(A.col_idx).to(dev)
    val = torch.from_numpy(A.vals).to(dev)
    X = torch.from_numpy(synth.vector(A.n * k, synth.DIST_NORMAL, 0, synth.STREAM_X, A.dtype)).to(dev).view(A.n, k)
    Y = torch.zeros((A.m, k), dtype=vt, device=dev)
    stream = torch.cuda.current_stream(dev)
    plan = lb.Plan(rp, col, val, A.n, kernel=args.kernel, with_spmm=True)
    spmm_path = spmm_path_of(plan.info(), k, s, A.row_ptr)
    for _ in range(args.warmup):
        plan.execute_multi(X, Y, W.alpha, W.beta, stream)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.15 if sampler else 0)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for a, b in ev:
        a.record(stream)
        plan.execute_multi(X, Y, W.alpha, W.beta, stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop(t0, time.time()) if sampler else None
    per = np.array([a.elapsed_time(b) for a, b in ev]) * 1e3
    plan.close()
    if rank != 0:
        return None
    med = float(np.median(per))
    bytes_ = A.nnz * (4 + s) + (A.m + 1) * 4 + A.n * k * s + A.m * k * s * (2 if W.beta != 0 else 1)
    peak, peak_kind = measured_peak()
    achieved = bytes_ / (float(per.mean()) * 1e-6) / 1e9
    return {
        "metric": f"CSR SpMM GFLOP/s (2*nnz*k per product, k={k})", "value": round(2.0 * A.nnz * k / (med * 1e-6) / 1e9, 2),
        "unit": "GFLOP/s", "n_gpus": 1, "steps": K, "warmup": args.warmup, "median_us": round(med, 2),
        "higher_is_better": True, "dtype": A.dtype, "data": "synthetic",
        "config": {"workload": workload_name, "k": k, "kernel": spmm_path[0], "launches_per_product": spmm_path[1]},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} copy bandwidth",
                     "algorithmic_bytes_per_product": int(bytes_), "traffic": None},
        "clocks": clocks,
    }


def run_spgemm(args, workload_name: str) -> dict | None:
    """C = A*A on the workload's matrix (the squared-matrix benchmark of
    OpSparse): the symbolic phase (handle creation: checks, binning, row
    sizes) timed on the host around a synchronised call, the numeric phase
    with CUDA events.  GFLOP/s = 2 * products / numeric time, products = the
    intermediate products a*b of Gustavson's method."""
    import torch
    import load_balanced_csr_gb300 as lb

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    A = synth.workload(workload_name, scale=args.scale).A
    s = A.vals.dtype.itemsize
    rp = torch.from_numpy(A.row_ptr).to(dev)
    col = torch.from_numpy(A.col_idx).to(dev)
    val = torch.from_numpy(A.vals).to(dev)
    stream = torch.cuda.current_stream(dev)
    sym = []
    for _ in range(3):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        h = lb.SpGEMM(rp, col, rp, col, A.n, val.dtype, stream=stream)
        sym.append((time.perf_counter() - t0) * 1e3)
        if _ < 2:
            h.close()
    out = h.compute(val, val, stream=stream)
    for _ in range(args.warmup):
        h.compute(val, val, out=out, stream=stream)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.15 if sampler else 0)
    K = min(args.steps, 30)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t0 = time.time()
    for a, b in ev:
        a.record(stream)
        h.compute(val, val, out=out, stream=stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop(t0, time.time()) if sampler else None
    per = np.array([a.elapsed_time(b) for a, b in ev]) * 1e3
    info = h.info()
    status = h.device_status()
    h.close()
    if rank != 0:
        return None
    med = float(np.median(per))
    products = info["products"]
    # compulsory bytes of the numeric phase: A and B read once, C written once
    bytes_ = 2 * (A.nnz * (4 + s) + (A.m + 1) * 4) + info["c_nnz"] * (4 + s) + (A.m + 1) * 4
    peak, peak_kind = measured_peak()
    achieved = bytes_ / (float(per.mean()) * 1e-6) / 1e9
    return {
        "metric": "SpGEMM C = A*A GFLOP/s (2 * intermediate products / numeric phase)",
        "value": round(2.0 * products / (med * 1e-6) / 1e9, 2), "unit": "GFLOP/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "median_us": round(med, 1), "higher_is_better": True, "dtype": A.dtype,
        "data": "synthetic",
        "config": {"workload": workload_name, "scale": args.scale, "products": products, "c_nnz": info["c_nnz"],
                   "bin_rows": info["bin_rows"], "numeric_bin_rows": info["numeric_bin_rows"],
                   "dense_slots": info["dense_slots"],
                   "dense_pieces": info["dense_pieces"], "dense_waves": info["dense_waves"],
                   "launches_per_compute": info["launches_per_compute"],
                   "symbolic_ms_median": round(float(np.median(sym)), 2), "device_status": status},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} copy bandwidth",
                     "algorithmic_bytes_per_product": int(bytes_), "traffic": None},
        "clocks": clocks,
    }


def run_gather(args, workload_name: str) -> dict | None:
    """Ceilings of the x gather on the workload's column pattern, by load
    path (spmv_gather_ceiling): the columns and the gathered values only, no
    matrix values, no floating-point work.  Each path is timed with CUDA
    events over args.steps launches after args.warmup; `gathers_per_sm_clk`
    divides the gathers by the SM count and the sampled SM clock."""
    import torch
    import load_balanced_csr_gb300 as lb

    rank, world, local = dist_env()
    if rank != 0:
        return None
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    W = synth.workload(workload_name)
    A = W.A
    col = torch.from_numpy(A.col_idx).to(dev)
    vals = torch.from_numpy(A.vals).to(dev)
    x = torch.from_numpy(W.x).to(dev)
    stream = torch.cuda.current_stream(dev)
    ut = np.uint64 if A.dtype == "f64" else np.uint32
    want = int(np.sum(W.x.view(ut)[A.col_idx].astype(np.uint64), dtype=np.uint64))
    want_vals = (want + int(np.sum(A.vals.view(ut).astype(np.uint64), dtype=np.uint64))) & (2**64 - 1)
    want_stream = int(np.sum(A.col_idx.astype(np.uint64), dtype=np.uint64))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    res = {}
    sampler = ClockSampler(local)
    time.sleep(0.15)
    t0 = time.time()
    for path in lb.GATHER_PATHS:
        cs = torch.zeros(1, dtype=torch.int64, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        lb.gather_ceiling(path, col, x, cs, err, stream, vals=vals)
        torch.cuda.synchronize(dev)
        expect = want_stream if path == "stream" else want_vals if path in lb.GATHER_WITH_VALUES else want
        ok = (int(cs.item()) & (2**64 - 1)) == expect and int(err.item()) == 0
        for _ in range(args.warmup):
            lb.gather_ceiling(path, col, x, cs, err, stream, vals=vals)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        torch.cuda.synchronize(dev)
        for a, b in ev:
            a.record(stream)
            lb.gather_ceiling(path, col, x, cs, err, stream, vals=vals)
            b.record(stream)
        torch.cuda.synchronize(dev)
        per = np.array([a.elapsed_time(b) for a, b in ev]) * 1e3
        res[path] = {"median_us": round(float(np.median(per)), 2), "checksum_ok": bool(ok)}
    clocks = sampler.stop(t0, time.time())
    mhz = clocks.get("sm_mhz") or 2070.0
    for path, r in res.items():
        if path != "stream":
            r["gathers_per_sm_clk"] = round(A.nnz / (r["median_us"] * 1e-6) / (sms * mhz * 1e6), 3)
    return {"metric": "x-gather ceiling by load path (columns + gathers only)", "unit": "us",
            "higher_is_better": False, "dtype": A.dtype, "data": "synthetic",
            "config": {"workload": workload_name, "nnz": A.nnz, "n": A.n, "steps": args.steps,
                       "warmup": args.warmup, "sms": sms},
            "paths": res, "clocks": clocks}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=synth.WORKLOADS)
    ap.add_argument("--all", action="store_true", help="one line per workload")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kernel", default="auto")
    ap.add_argument("--ipt", type=int, default=0)
    ap.add_argument("--group", type=int, default=0, help="Row-grouped CSR group size (0 = plan's choice)")
    ap.add_argument("--long-min", type=int, default=0, help="long-row threshold (0 = plan's default)")
    ap.add_argument("--rhs", type=int, default=0, help="k > 0: time SpMM with k right-hand sides instead")
    ap.add_argument("--transposed", action="store_true", help="time the transposed product A^T x instead")
    ap.add_argument("--spgemm", action="store_true", help="time SpGEMM C = A*A instead")
    ap.add_argument("--gather-only", action="store_true",
                    help="time the x gather alone on the workload's columns, by load path")
    ap.add_argument("--scale", type=int, default=1,
                    help="SpGEMM only: shrink the workload by this factor (small cases for profiling)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload block (default run, N = 1 only)")
    ap.add_argument("--per-config-cpu-budget", type=float, default=3.0,
                    help="seconds of oracle time per workload in the per-config block")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank, world, _ = dist_env()
    if args.impl == "reference":
        for name in (synth.WORKLOADS if args.all else [args.workload]):
            out = run_reference(args, name)
            if out is not None:
                print(json.dumps(out), flush=True)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    names = synth.WORKLOADS if args.all else [args.workload]
    for name in names:
        if args.gather_only:
            out = run_gather(args, name)
            if out is not None:
                print(json.dumps(out), flush=True)
            continue
        out = run_spgemm(args, name) if args.spgemm else run_spmm(args, name) if args.rhs > 0 else \
            run_gpu(args, name)
        if out is not None:
            # the oracle is timed on rank 0 at N = 1 only
            out["cpu_baseline"] = cpu_baseline_leg(name, args.cpu_budget) \
                if world == 1 and not args.no_cpu_baseline and not args.spgemm else None
            out["source_hash"] = kernel_source_hash()
            if world == 1 and not args.no_per_config and not args.all and args.rhs == 0 and not args.spgemm \
                    and not args.transposed and args.kernel == "auto":
                out["per_config"] = run_per_config(args)
            print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
