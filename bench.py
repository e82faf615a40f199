"""Benchmark of the autotuned matmul on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--report]

A step is one warm pass of the hot path: mm_autotune_execute on one set of
inputs already resident in HBM (key, table lookup, one launch of the tuned
kernel).  The first call on an empty table is the cold tune and is timed
separately, as is the host latency of a cache hit.  Inputs rotate over enough
sets to exceed twice the L2 size, so no step reads the previous step's
inputs from L2.  One JSON line is printed by rank 0.

--impl reference times the CPU oracle (fp64 triple loop) on the same
workload, each step a bounded sample of output elements.
--report prints one line per named workload (not the driver's contract).
--candidate NAME runs one candidate directly instead of the tuner (profiling).
"""
from __future__ import annotations

import argparse
import ctypes
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

BF16, F16, F32 = synth.BF16, synth.F16, synth.F32

# name -> (M, N, K, layout, (dtA, dtB, dtC), distA, distB, lda_pad, batch, seed)
WORKLOADS = {
    "square_4096_bf16": (4096, 4096, 4096, "NN", (BF16, BF16, BF16), "normal", "normal", 0, 1, 1002),
    "square_4096_bf16_nt": (4096, 4096, 4096, "NT", (BF16, BF16, BF16), "normal", "normal", 0, 1, 1002),
    "square_4096_bf16_tn": (4096, 4096, 4096, "TN", (BF16, BF16, BF16), "normal", "normal", 0, 1, 1002),
    "square_4096_bf16_tt": (4096, 4096, 4096, "TT", (BF16, BF16, BF16), "normal", "normal", 0, 1, 1002),
    "square_8192_bf16": (8192, 8192, 8192, "NN", (BF16, BF16, BF16), "normal", "normal", 0, 1, 1002),
    "small_256_bf16": (256, 256, 256, "NN", (BF16, BF16, F32), "u11", "u11", 0, 1, 1000),
    "gemv_m1_4096_bf16": (1, 4096, 4096, "NN", (BF16, BF16, BF16), "normal", "normal:0.02", 0, 1, 1001),
    "gemv_m8_4096_bf16": (8, 4096, 4096, "NN", (BF16, BF16, BF16), "normal", "normal:0.02", 0, 1, 1001),
    "gemv_m16_4096_bf16": (16, 4096, 4096, "NN", (BF16, BF16, BF16), "normal", "normal:0.02", 0, 1, 1001),
    "skinny_25088x4096x64_f32_nt": (25088, 4096, 64, "NT", (F32, F32, F32), "u11", "u11", 0, 1, 1003),
    "skinny_4096x4096x64_f32_nt": (4096, 4096, 64, "NT", (F32, F32, F32), "u11", "u11", 0, 1, 1003),
    "splitk_128x128x65536_bf16": (128, 128, 65536, "NN", (BF16, BF16, BF16), "u11", "u11", 0, 1, 1003),
    "batched_32x512_bf16": (512, 512, 512, "NN", (BF16, BF16, F32), "normal", "normal", 0, 32, 1004),
}
for _m in (1, 16, 127, 1000, 4097, 8192):
    for _t in ("N", "T"):
        WORKLOADS[f"bucket_m{_m}_lda4100_{_t.lower()}_bf16"] = (
            _m, 4096, 4096, "N" + _t, (BF16, BF16, BF16), "normal", "normal", 4, 1, 1004)

DEFAULT_WORKLOAD = "square_4096_bf16"
GEMV_WORKLOAD = "gemv_m1_4096_bf16"
# configurations whose oracle is also timed on a single core
SINGLE_THREAD_BASELINE = ("small_256_bf16", "gemv_m1_4096_bf16", "gemv_m8_4096_bf16",
                          "gemv_m16_4096_bf16")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def workload_shape(name):
    M, N, K, lay, dt, da, db, pad, batch, seed = WORKLOADS[name]
    return dict(M=M, N=N, K=K, layout=lay, dt=dt, dist_a=da, dist_b=db, pad=pad, batch=batch,
                seed=seed)


def make_host_inputs(w):
    at, bt = w["layout"][0] == "T", w["layout"][1] == "T"
    M, N, K, batch = w["M"], w["N"], w["K"], w["batch"]
    lda = (M if at else K) + w["pad"]
    ldb = K if bt else N
    A = synth.make_operand(w["seed"], w["dt"][0], M, K, ld=lda, trans=at, batch=batch,
                           dist=w["dist_a"])
    B = synth.make_operand(w["seed"] + 1, w["dt"][1], K, N, ld=ldb, trans=bt, batch=batch,
                           dist=w["dist_b"])
    C = synth.output_buffer(w["dt"][2], M, N, batch=batch)
    return A, B, C


def workload_config(w, name, n_gpus):
    """The `config` object of a line: the same keys for both arms."""
    return {"workload": name, "M": w["M"], "N": w["N"], "K": w["K"], "layout": w["layout"],
            "batch": w["batch"],
            "lda": (w["M"] if w["layout"][0] == "T" else w["K"]) + w["pad"],
            "dtypes": [synth.DTYPE_NAMES[x] for x in w["dt"]],
            "parallelism": f"replicas{n_gpus}",
            "l2": "inputs rotate over sets totalling more than 2 x L2 between steps"}


def algorithmic(w):
    eb = synth.DTYPE_BYTES
    M, N, K, b = w["M"], w["N"], w["K"], w["batch"]
    flops = 2.0 * M * N * K * b
    nbytes = float((M * K * eb[w["dt"][0]] + K * N * eb[w["dt"][1]] + M * N * eb[w["dt"][2]]) * b)
    return flops, nbytes


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.close()
        rows = []
        with open(self.file.name) as f:
            for r in csv.reader(io.StringIO(f.read())):
                if len(r) >= 9:
                    rows.append([x.strip() for x in r])
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------- CPU oracle
def oracle_rate(A, B, w, budget_s, seed=7):
    """Time the oracle on a bounded sample of output elements; returns
    (TFLOP/s, seconds, points)."""
    import oracle
    rng = np.random.default_rng(seed)
    M, N, K, batch = w["M"], w["N"], w["K"], w["batch"]

    def pts(n):
        return np.stack([rng.integers(0, batch, n), rng.integers(0, M, n),
                         rng.integers(0, N, n)], axis=1)

    n = 64
    t0 = time.perf_counter()
    oracle.gemm_points(A, B, K, pts(n))
    dt = max(time.perf_counter() - t0, 1e-6)
    n = int(max(64, min(5e7, n * budget_s / dt)))
    t0 = time.perf_counter()
    oracle.gemm_points(A, B, K, pts(n))
    dt = time.perf_counter() - t0
    return 2.0 * n * K / dt / 1e12, dt, n


def run_reference(args, w, name):
    import oracle
    oracle.build()
    A, B, _ = make_host_inputs(w)
    cores = oracle.num_threads()
    # size one step so the whole run stays within ~2 minutes
    total_steps = args.steps + args.warmup
    per_step_s = max(0.05, min(10.0, 120.0 / max(total_steps, 1)))
    rate, dt, npts = oracle_rate(A, B, w, per_step_s)
    rng = np.random.default_rng(11)
    M, N, K, batch = w["M"], w["N"], w["K"], w["batch"]

    def step():
        p = np.stack([rng.integers(0, batch, npts), rng.integers(0, M, npts),
                      rng.integers(0, N, npts)], axis=1)
        oracle.gemm_points(A, B, K, p)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = time.perf_counter() - t0
    value = 2.0 * npts * K * args.steps / t / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": workload_config(w, name, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{npts} random output elements per step (K={K} each)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU bench
METRIC = "tuned GEMM TFLOP/s & % of roofline at 1 GB300; cold-tune and cache-hit ms"


def max_over_ranks(x, world, device):
    """The largest of a per-rank number over all ranks (the job ends when its
    slowest replica does); x itself at world 1."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(work_per_rank, world, seconds):
    """Whole-job throughput: every replica does the same work (weak scaling),
    timed by the slowest rank."""
    return work_per_rank * world / seconds


def ensure_built():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_mm_build", os.path.join(ROOT, "matmul_selection_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()


def kernel_sources(kernel_name):
    """The source files that hold a candidate's kernels."""
    kdir = os.path.join(ROOT, "matmul_selection_gb300", "csrc", "kernels")
    if kernel_name.startswith(("tc_repack", "tc2_repack", "gemv_swap_tc_repack")):
        names = ["repack.cu", "tc_gemm.cu"]
    elif kernel_name.startswith(("tc", "gemv_swap_tc")):
        names = ["tc_gemm.cu"]
    elif kernel_name in ("gemv_n_cluster", "gemv_t_rows", "gemv_n_stream", "gemv_t_stream"):
        names = ["gemv_fast.cu"]
    elif kernel_name in ("gemv_n_mma", "gemv_t_mma"):
        names = ["gemv_mma.cu"]
    elif kernel_name.startswith("gemv"):
        names = ["gemv.cu"]
    else:
        names = ["naive.cu"]
    return [os.path.join(kdir, n) for n in names]


def sources_sha1(kernel_name):
    import hashlib
    h = hashlib.sha1()
    for path in kernel_sources(kernel_name):
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def traffic_for(kernel_name, workload):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(f"{kernel_name}@{workload}")
    if not e or e.get("source_sha1") != sources_sha1(kernel_name):
        return None
    return e.get("dram_bytes_per_launch")


def run_ours(args, w, name, rank, world, peaks, lite=False):
    """One workload through the library.  lite: only the cold tune, the warm
    timed loop and the roofline (no cache-hit latency loop, no clock record,
    no end-to-end leg), for a sub-record of the main line."""
    import torch

    import matmul_selection_gb300 as mm
    dev = torch.device("cuda", torch.cuda.current_device())
    mm.check(mm.mm_set_option("peak_tflops", str(peaks["bf16_tflops"])))
    mm.check(mm.mm_set_option("peak_gbs", str(peaks["hbm_gbs"])))
    M, N, K, batch = w["M"], w["N"], w["K"], w["batch"]
    A, B, C = make_host_inputs(w)
    flops, nbytes = algorithmic(w)
    set_bytes = A.buf.nbytes + B.buf.nbytes + C.buf.nbytes
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 << 20)
    R = max(2, math.ceil(2 * l2 / set_bytes))
    R = min(R, max(2, int(40e9 // set_bytes)))
    hA = torch.from_numpy(A.buf.view(np.uint8))
    hB = torch.from_numpy(B.buf.view(np.uint8))
    sets = []
    for r in range(R):
        dA = hA.to(dev)
        dB = hB.to(dev)
        dC = torch.empty(C.buf.nbytes, dtype=torch.uint8, device=dev)
        sets.append((dA, dB, dC))
    dt = w["dt"]
    b = None if batch == 1 else (batch, A.bstride, B.bstride, C.bstride)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    forced = args.candidate
    if forced:
        idx = mm.candidate_names().index(forced)

    # arguments converted to C types once, so a step costs one foreign call
    lib = mm.library_handle()
    cdt = mm.mm_dtypes(*dt)
    clay = mm.LAYOUTS[w["layout"]]
    cb = None if b is None else ctypes.byref(mm.mm_batch(*b))
    ptrs = [(s_[0].data_ptr(), s_[1].data_ptr(), s_[2].data_ptr()) for s_ in sets]

    def call(s):
        pa, pb, pc = ptrs[s % R]
        if forced:
            return lib.mm_execute_candidate(idx, pa, pb, pc, M, N, K, A.ld, B.ld, C.ld, cdt, clay,
                                            cb, sh)
        return lib.mm_autotune_execute(pa, pb, pc, M, N, K, A.ld, B.ld, C.ld, cdt, clay, cb, sh)

    torch.cuda.synchronize()
    # the roofline probes run once per device (first call or first tune):
    # timed here on their own, so the cold tune below has them warm
    t0 = time.perf_counter()
    mm.check(mm.mm_device_peaks()[0])
    probe_ms = (time.perf_counter() - t0) * 1e3
    mm.mm_cache_clear()
    cold_ms = hit_ms = None
    if forced:
        mm.check(call(0))
        winner = forced
    else:
        # cold tune: the first call on an empty table
        t0 = time.perf_counter()
        mm.check(call(0))
        torch.cuda.synchronize()
        cold_ms = (time.perf_counter() - t0) * 1e3
        st = mm.mm_tune_key(M, N, K, A.ld, B.ld, C.ld, dt, w["layout"], b)
        winner = mm.mm_candidate_name(mm.mm_lookup(st[1])[1])
        # warm cache-hit latency: host wall time of call + sync
        hits = []
        for i in range(100 if lite else 200 if args.report else 1000):
            t0 = time.perf_counter()
            call(i)
            torch.cuda.synchronize()
            hits.append((time.perf_counter() - t0) * 1e3)
        hit_ms = statistics.median(hits)
    # host time to enqueue one warm call (no synchronisation)
    torch.cuda.synchronize()
    enq = []
    for i in range(200):
        t0 = time.perf_counter()
        call(i)
        enq.append((time.perf_counter() - t0) * 1e6)
    torch.cuda.synchronize()
    enqueue_us = statistics.median(enq)
    # timed region
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if not lite:
        # the clock sampler (an nvidia-smi process polling every 200 ms) starts
        # first; the timed region is then a burst, so its denominator is the
        # burst peak, and the sustained rate is taken separately below
        sampler.start()
        time.sleep(0.3)
    for i in range(args.warmup):
        mm.check(call(i))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = mm.mm_get_stats()["launches"]
    ev0.record(stream)
    for i in range(args.steps):
        call(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    launches = mm.mm_get_stats()["launches"] - launches0
    if world > 1:
        torch.distributed.barrier()
    # the sampler polls every 200 ms and a timed region of a few steps is far
    # shorter: keep the same workload running for about a second more so that
    # the clock record reflects this load; its chunks are timed too, and those
    # of the second half give the sustained rate (the power cap settles within
    # a fraction of a second of continuous load)
    t_hold = time.perf_counter()
    i = 0
    chunks = []
    while not lite and time.perf_counter() - t_hold < 1.0:
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(50):
            call(i)
            i += 1
        c1.record(stream)
        torch.cuda.synchronize()
        chunks.append((time.perf_counter() - t_hold, c0, c1))
    clocks = None
    sustained = None
    if not lite:
        clocks = sampler.stop()
        clocks["window"] = ("0.3 s idle while the sampler starts, the timed region, and 1 s of "
                            "the same calls after it")
        late = [c for c in chunks if c[0] >= 0.5]
        if late:
            ms = sum(c0.elapsed_time(c1) for _, c0, c1 in late)
            n_calls = 50 * len(late)
            sustained = {"ms_per_step": ms / n_calls, "steps": n_calls,
                         "window": "the second half of 1 s of back-to-back calls after the "
                                   "timed region (chunks of 50, each timed by events)"}
    total_ms = ev0.elapsed_time(ev1)
    # every warm step is one call of the tuned candidate: its mean device time
    # per launch is the timed loop's device time over the steps
    kern_ms = total_ms / args.steps
    total_ms = max_over_ranks(total_ms, world, dev)
    value = aggregate_rate(flops * args.steps, world, total_ms * 1e-3) / 1e12
    # context only: the vendor library on the same shape and rotating inputs
    cublas_tflops = None
    if args.cublas and batch == 1 and not w["pad"] and dt[0] == dt[1] and dt[0] != F32:
        tdt = {BF16: torch.bfloat16, F16: torch.float16}[dt[0]]
        tA = [x[0].view(tdt).view(M, K) if w["layout"][0] == "N" else x[0].view(tdt).view(K, M).t()
              for x in sets]
        tB = [x[1].view(tdt).view(K, N) if w["layout"][1] == "N" else x[1].view(tdt).view(N, K).t()
              for x in sets]
        # timed as the library's burst is: after a 0.3 s pause, 5 warm-up calls
        torch.cuda.synchronize()
        time.sleep(0.3)
        for i in range(5):
            torch.matmul(tA[i % R], tB[i % R])
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        nrep = args.steps
        for i in range(nrep):
            torch.matmul(tA[i % R], tB[i % R])
        e1.record(stream)
        torch.cuda.synchronize()
        cublas_tflops = flops * nrep / (e0.elapsed_time(e1) * 1e-3) / 1e12
    # end to end from pinned host buffers through the host entry point
    e2e = None
    if not lite:
        e2e_steps = max(1, min(args.steps, 50))
        pA = torch.empty(A.buf.nbytes, dtype=torch.uint8, pin_memory=True)
        pB = torch.empty(B.buf.nbytes, dtype=torch.uint8, pin_memory=True)
        pC = torch.empty(C.buf.nbytes, dtype=torch.uint8, pin_memory=True)
        pA.copy_(hA)
        pB.copy_(hB)
        mm.check(mm.mm_autotune_execute_host(pA.data_ptr(), pB.data_ptr(), pC.data_ptr(), M, N,
                                             K, A.ld, B.ld, C.ld, dt, w["layout"], b, sh))
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            mm.check(mm.mm_autotune_execute_host(pA.data_ptr(), pB.data_ptr(), pC.data_ptr(), M,
                                                 N, K, A.ld, B.ld, C.ld, dt, w["layout"], b, sh))
        e2e_s = time.perf_counter() - t0
        e2e_s = max_over_ranks(e2e_s, world, dev)
        e2e = {"value": aggregate_rate(flops * e2e_steps, world, e2e_s) / 1e12, "unit": "TFLOP/s",
               "steps": e2e_steps, "h2d_bytes_per_step": int(A.buf.nbytes + B.buf.nbytes),
               "d2h_bytes_per_step": int(M * N * batch * synth.DTYPE_BYTES[dt[2]])}
    # roofline of the dominant (tuned) kernel: the bound is whichever of the
    # memory time (algorithmic bytes / HBM peak) and the compute time
    # (flops / tensor peak) is longer
    tf32 = dt[0] == F32
    tensor_peak = peaks["bf16_tflops"] * (1.1 / 2.25 if tf32 else 1.0)
    hbm = nbytes / (peaks["hbm_gbs"] * 1e9) > flops / (tensor_peak * 1e12)
    if hbm:
        achieved = nbytes / (kern_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic_for(winner, name),
                "peak_source": peaks["source"], "algorithmic_bytes": nbytes}
    else:
        achieved = flops / (kern_ms * 1e-3) / 1e12
        peak = tensor_peak
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic_for(winner, name),
                "peak_source": peaks["source"] + (" x tf32/bf16 nominal ratio" if tf32 else ""),
                "algorithmic_flops": flops}
    roof["kernel"] = winner
    roof["kernel_ms"] = kern_ms
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {BF16: "bf16", F16: "f16", F32: "f32"}[dt[0]], "data": "synthetic",
        "config": workload_config(w, name, world),
        "rotation": f"{R} input sets of {set_bytes / 1e6:.1f} MB",
        "winner": winner, "cold_tune_ms": cold_ms, "cache_hit_ms": hit_ms,
        "peak_probe_ms": probe_ms,
        "host_enqueue_us": enqueue_us,
        "context_cublas_tflops": cublas_tflops,
        "gpu_launches": int(launches), "clocks": clocks, "roofline": roof, "e2e": e2e,
    }
    if hbm:
        line["gbs"] = nbytes * args.steps * world / (total_ms * 1e-3) / 1e9
    if sustained is not None:
        t = sustained["ms_per_step"] * 1e-3
        if hbm:
            sustained.update(value=nbytes / t / 1e9, unit="GB/s", peak=peaks["hbm_gbs"],
                             peak_source=peaks["source"] + " (copy bandwidth)")
        else:
            sp = peaks["bf16_tflops_sustained"] * (1.1 / 2.25 if tf32 else 1.0)
            sustained.update(value=flops / t / 1e12, unit="TFLOP/s", peak=sp,
                             peak_source=peaks["source"] + " sustained")
        sustained["frac"] = sustained["value"] / sustained["peak"]
        line["sustained"] = sustained
    return line, (A, B)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--report", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--cublas", action="store_true",
                    help="also time torch.matmul on the same shape (context, not a target)")
    ap.add_argument("--only", default=None, help="with --report: comma-separated name filters")
    ap.add_argument("--candidate", default=None,
                    help="run this candidate directly (no tuning); for profiling")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = workload_shape(args.workload)
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w, args.workload)
        return
    ensure_built()
    import torch
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    peaks = load_peaks()
    names = sorted(WORKLOADS) if args.report else [args.workload]
    if args.only:
        names = [n for n in names if any(o in n for o in args.only.split(","))]
    for name in names:
        wl = workload_shape(name)
        steps = args.steps
        if args.report:
            args.steps = min(steps, 200)
        line, (A, B) = run_ours(args, wl, name, rank, world, peaks)
        args.steps = steps
        if name == DEFAULT_WORKLOAD and not args.report and not args.candidate:
            # the second target's workload, timed the same way, as a sub-record
            args.steps = max(steps, 200)
            g, _ = run_ours(args, workload_shape(GEMV_WORKLOAD), GEMV_WORKLOAD, rank, world, peaks,
                            lite=True)
            args.steps = steps
            r = g["roofline"]
            line["gemv_m1"] = {"workload": GEMV_WORKLOAD, "winner": g["winner"],
                               "kernel_us": r["kernel_ms"] * 1e3, "value_gbs": r["achieved"],
                               "frac": r["frac"], "peak_gbs": r["peak"], "bound": r["bound"],
                               "steps": max(steps, 200),
                               "cold_tune_ms": g["cold_tune_ms"],
                               "cache_hit_ms": g["cache_hit_ms"],
                               "gpu_launches": g["gpu_launches"],
                               "traffic": r["traffic"]}
        if rank == 0:
            import oracle
            oracle.build()
            rate, dt, npts = oracle_rate(A, B, wl, 2.0 if args.report else args.cpu_budget_s)
            cores = oracle.num_threads()
            line["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s", "cores": cores,
                                    "kind": "oracle",
                                    "sample": f"{npts} random output elements (K={wl['K']} each),"
                                              f" {dt:.1f} s"}
            if name in SINGLE_THREAD_BASELINE and cores > 1:
                # the small and GEMV configurations are also timed on one core
                oracle.set_num_threads(1)
                try:
                    r1, dt1, n1 = oracle_rate(A, B, wl, 1.0 if args.report else 2.0)
                finally:
                    oracle.set_num_threads(cores)
                line["cpu_baseline_1core"] = {
                    "value": r1, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                    "sample": f"{n1} random output elements (K={wl['K']} each), {dt1:.1f} s"}
            print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
