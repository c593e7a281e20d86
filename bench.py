#!/usr/bin/env python3
"""Benchmark: SGEMM TFLOP/s at 4096^3 fp32 and % of the GB300 FP32 FFMA peak.

One step = one sgemm() call (the library's public entry point, path chosen by
its selector) on the 4096 x 4096 x 4096 row-major NN problem, alpha = 1,
beta = 0, A and B uniform[-1, 1] from seed 3, inputs resident in HBM.  L2 is
flushed between steps by writing a 256 MB buffer; the flush is outside the
CUDA events that time each step.

Prints ONE JSON line (rank 0).  The headline value comes from K steps with
nothing but the calls in them.  Keys beyond the base contract:
  roofline      dominant kernel: achieved / peak, its launches timed by the
                library's CUDA event pair on the launching stream over a
                second region of the same K steps (FFMA: "alu" bound, peak =
                SMs x 128 lanes x 2 flop x max SM clock; tensor cores: the
                measured bf16 peak x 1.1/2.25, and beside it SMs x the
                measured kind::tf32 MAC rate per clock (library probe) x 2 x
                SM clock), DRAM traffic from the committed ncu summary when
                it matches the current kernel.
  cpu_baseline  the CPU oracle (fp64 triple loop) timed on a bounded sample
                of the same workload on the host cores.
  e2e           the same metric through sgemm_host() on pinned host
                buffers: the library's H2D of A and B, the GEMM and the D2H
                of C (pipelined in row blocks), all inside the timed region.
  paths         every GPU path timed on the same workload (TFLOP/s, fraction
                of its roofline, error vs the oracle on sample points).
  workloads     every workload through sgemm(): flushed median and min,
                unflushed median, roofline fraction, and the CPU oracle's
                GFLOP/s on a bounded row sample (all cores; one core for the
                small square ones) with the GPU/oracle speed-up.
  clocks        nvidia-smi SM clock samples during the timed region.

--impl reference times the CPU oracle itself (the reference arm).
Under torchrun (N > 1) every rank runs an independent replica (the
problem is not sharded); value = all ranks' flops / max rank time.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gemm_inputs as gi  # noqa: E402

METRIC = "SGEMM TFLOP/s at 4096^3 fp32 and % of GB300 FP32 FFMA peak (1 GPU)"
UNIT = "TFLOP/s"
WORKLOAD = gi.HEADLINE
FLUSH_BYTES = 256 << 20
FP32_LANES_PER_SM = 128


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 25 ms) of SM clock and throttle reasons; each
    sample carries its host arrival time so that only those taken inside the
    timed region count."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen in samples that
        arrived within [t0, t1] (host perf_counter; all samples if None)."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if t0 is not None and not (t0 <= ts <= t1):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ helpers
def job_throughput(local_ms: float, steps: int, flops_per_step: float, device=None):
    """(max over ranks of the timed milliseconds, whole-job TFLOP/s).

    Every rank runs an independent replica of the step; the job takes as long
    as its slowest rank, and it did world * steps steps in that time.  Works
    with any torch.distributed backend (NCCL on GPUs, gloo in the CPU tests);
    without an initialised process group it is the single-rank value.
    """
    import torch
    import torch.distributed as dist
    world = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    t = float(local_ms)
    if world > 1:
        x = torch.tensor([t], dtype=torch.float64, device=device)
        dist.all_reduce(x, op=dist.ReduceOp.MAX)
        t = float(x.item())
    return t, world * steps * flops_per_step / (t / 1e3) / 1e12


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}, "fallback"


def kernel_source_sha(files):
    """Short sha of a kernel's own source files (as profiles/traffic.json keys them)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp32_gemm_05_gb300", "csrc")
    for fn in files:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel_key: str):
    """DRAM bytes (read + write) per launch of `kernel_key` from
    profiles/traffic.json, if that ncu capture was taken on the kernel's
    current source files; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        tab = json.load(f)
    ent = tab.get(kernel_key)
    if not ent:
        return None
    try:
        if ent.get("source_sha") != kernel_source_sha(ent["files"]):
            return None
    except OSError:
        return None
    return ent["dram_bytes_per_launch"]


def oracle_sample(w, A, B, C, seconds_target=12.0, max_rows=None):
    """Times the CPU oracle on whole rows of C (bounded sample).

    Returns (flops_per_s, rows, seconds, threads).
    """
    import oracle
    oracle.build()
    threads = oracle.num_threads()

    def run(rows):
        r = np.repeat(np.arange(rows, dtype=np.int64), w.N)
        c = np.tile(np.arange(w.N, dtype=np.int64), rows)
        t0 = time.perf_counter()
        oracle.gemm_f64(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A, A.shape[1], B,
                        B.shape[1], w.beta, C, w.N, points=(r, c))
        return time.perf_counter() - t0

    probe_rows = max(1, threads // 4)
    dt = run(probe_rows)
    per_row = max(dt / probe_rows, 1e-6)
    rows = int(max(1, min(w.M, seconds_target / per_row)))
    if max_rows:
        rows = min(rows, max_rows)
    dt = run(rows)
    flops = 2.0 * rows * w.N * w.K
    return flops / dt, rows, dt, threads


# ------------------------------------------------------------------ reference arm
def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = gi.WORKLOADS[WORKLOAD]
    A, B, C = gi.make_inputs(w)
    # size each step so the whole run stays near 2.5 minutes of CPU time
    per_step = max(1.0, min(args.ref_seconds, 150.0 / (args.steps + 0.25 * args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, A, B, C, seconds_target=per_step / 4)
    vals, rows_l, secs = [], [], []
    for _ in range(args.steps):
        v, rows, dt, threads = oracle_sample(w, A, B, C, seconds_target=per_step)
        vals.append(v)
        rows_l.append(rows)
        secs.append(dt)
    value = sum(2.0 * r * w.N * w.K for r in rows_l) / sum(secs) / 1e12
    sample = (f"rows 0..{rows_l[-1] - 1} of C ({rows_l[-1]} x {w.N} outputs, "
              f"{2 * rows_l[-1] * w.N * w.K:.3e} flop per step) of the {w.M}x{w.N}x{w.K} NN problem")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * statistics.mean(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, flushed=False),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def event_times(call, stream, flush, reps, flushed):
    """CUDA-event durations (ms) of `reps` calls on `stream`; with `flushed`
    L2 is flushed before each call, outside its events."""
    import torch
    ev = []
    for i in range(reps):
        if flushed:
            flush.fill_(0.25 + i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


# 1-core oracle timings for these workloads (the small square ones)
ONE_CORE = ("sq256_nn", "sq1024_nn", "sq2048_nn_ab")


def workload_table(dev, stream, flush, ffma_peak, tf32_peak, hbm_gbs, reps=5, oracle_s=1.0):
    """Every workload through sgemm() (the selector's path), device-timed with
    L2 flushed between calls (median and min) and without flushing (median),
    against the roofline of the path that ran: attainable = min(the path's
    compute peak, arithmetic intensity x HBM).  Inputs are drawn on the device
    (seeded, the workload's distribution): this table times; the parity tests
    check.  With oracle_s > 0 the CPU oracle is timed beside each workload on
    a bounded sample of whole rows of C (its own numpy draw), on all host
    cores and, for the small square workloads, on one core."""
    import torch
    import dense_fp32_gemm_05_gb300 as sg

    names = {sg.PATH_FFMA: "ffma", sg.PATH_3XTF32: "3xtf32", sg.PATH_TF32: "tf32",
             sg.PATH_GEMV: "gemv"}
    table = {}
    for name, w in gi.WORKLOADS.items():
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed)
        sa, sb, sc = w.stored_shapes()

        def draw(shape):
            if w.dist == "uniform":
                return torch.rand(shape, generator=g, device=dev) * 2.0 - 1.0
            return torch.randn(shape, generator=g, device=dev) * w.std
        dA, dB = draw(sa), draw(sb)
        dC = draw(sc) if w.beta != 0 else torch.zeros(sc, device=dev)
        st, plan = sg.sgemm_plan_detail(w.transA, w.transB, w.M, w.N, w.K, sa[1], sb[1], w.N)
        path = names.get(plan["path"], str(plan["path"])) if st == 0 else "?"
        # the thin path's tensor-core form (128 columns per CTA) runs 3xTF32
        thin_tc = st == 0 and path == "gemv" and plan["tile_n"] == 128

        def call():
            st = sg.sgemm(w.transA, w.transB, w.M, w.N, w.K, w.alpha, dA.data_ptr(), sa[1],
                          dB.data_ptr(), sb[1], w.beta, dC.data_ptr(), w.N, stream)
            if st != 0:
                raise sg.SgemmError(st)
        call()
        torch.cuda.synchronize(dev)
        flushed = event_times(call, stream, flush, reps, True)
        warm = event_times(call, stream, flush, reps, False)
        ms = statistics.median(flushed)
        tfl = w.flops / (ms / 1e3) / 1e12
        gbs = w.compulsory_bytes() / (ms / 1e3) / 1e9
        compute = {"ffma": ffma_peak, "gemv": tf32_peak / 3.0 if thin_tc else ffma_peak,
                   "3xtf32": tf32_peak / 3.0, "tf32": tf32_peak}.get(path, ffma_peak)
        hbm_roof = w.flops / w.compulsory_bytes() * hbm_gbs / 1e3
        attain = min(compute, hbm_roof)
        ent = {"path": path, "ms": round(ms, 4), "ms_min": round(min(flushed), 4),
               "ms_unflushed": round(statistics.median(warm), 4),
               "tflops": round(tfl, 3),
               "tflops_unflushed": round(w.flops / (statistics.median(warm) / 1e3) / 1e12, 3),
               "gbs": round(gbs, 1),
               "bound": "hbm" if hbm_roof < compute else
                        ("tensor" if path in ("3xtf32", "tf32") or thin_tc else "alu"),
               "attainable_tflops": round(attain, 3), "frac": round(tfl / attain, 4)}
        del dA, dB, dC
        if oracle_s > 0:
            A, B, C = gi.make_inputs(w)
            v, rows, dt, threads = oracle_sample(w, A, B, C, seconds_target=oracle_s)
            ent["oracle"] = {"gflops": round(v / 1e9, 3), "threads": threads, "rows": rows,
                             "seconds": round(dt, 2)}
            ent["speedup_vs_oracle"] = round(tfl * 1e12 / v, 1)
            if name in ONE_CORE:
                import oracle
                n = oracle.num_threads()
                oracle.set_num_threads(1)
                try:
                    v1, rows1, dt1, _ = oracle_sample(w, A, B, C, seconds_target=oracle_s)
                finally:
                    oracle.set_num_threads(n)
                ent["oracle_1core"] = {"gflops": round(v1 / 1e9, 3), "rows": rows1,
                                       "seconds": round(dt1, 2)}
            del A, B, C
        table[name] = ent
    torch.cuda.empty_cache()
    return table


def workload_config(w, flushed=True):
    cfg = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
           "layout": w.transA + w.transB, "alpha": w.alpha, "beta": w.beta,
           "dist": w.dist, "seed": w.seed, "storage": "row-major fp32"}
    if flushed:
        cfg["l2"] = f"flushed between steps ({FLUSH_BYTES >> 20} MB write, outside the timed events)"
    return cfg


# ------------------------------------------------------------------ GPU arm
def gpu_arm(args):
    import torch
    import dense_fp32_gemm_05_gb300 as sg
    from dense_fp32_gemm_05_gb300 import build as sgbuild

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sgbuild.build()
    sg.load()

    w = gi.WORKLOADS[WORKLOAD]
    A, B, C = gi.make_inputs(w)
    dA = torch.from_numpy(A).to(dev)
    dB = torch.from_numpy(B).to(dev)
    dC = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    lda, ldb, ldc = A.shape[1], B.shape[1], w.N

    def call(path=sg.PATH_AUTO, out=dC, a=dA, b=dB):
        st = sg.sgemm_ex(w.transA, w.transB, w.M, w.N, w.K, w.alpha, a.data_ptr(), lda,
                         b.data_ptr(), ldb, w.beta, out.data_ptr(), ldc, stream, path, 0)
        if st != 0:
            raise sg.SgemmError(st)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed_steps(n):
        """n steps, L2 flushed before each outside its events: per-step ms."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            flush.fill_(float(i))
            starts[i].record(stream)
            call()
            ends[i].record(stream)
        barrier()
        return [a.elapsed_time(b) for a, b in zip(starts, ends)]

    # ---- warm-up
    for _ in range(args.warmup):
        flush.fill_(1.0)
        call()
    torch.cuda.synchronize(dev)

    # ---- timed region: K steps, per-step CUDA events on the launching stream
    # (nothing else in the calls: the kernel timing hook is off here)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    launches0 = sg.sgemm_launch_count()
    t_begin = time.perf_counter()
    step_ms = timed_steps(args.steps)
    t_end = time.perf_counter()
    launches = sg.sgemm_launch_count() - launches0
    t_wall = t_end - t_begin
    total_ms, value = job_throughput(sum(step_ms), args.steps, w.flops, device=dev)
    ms_per_step = total_ms / args.steps

    # ---- roofline region: the same K steps again, now with the library's
    # CUDA event pair around each launch of the main kernel (on the launching
    # stream).  The events sit between the call's kernels, so this region's
    # call times are not the headline; its kernel times are the roofline's.
    sg.sgemm_timing_enable(args.steps)
    t_rbegin = time.perf_counter()
    hooked_ms = timed_steps(args.steps)
    t_rend = time.perf_counter()
    kernel_ms = sg.sgemm_timing_read(args.steps)
    sg.sgemm_timing_enable(0)
    time.sleep(0.05)                # the last in-region sample reaches the reader
    sampler.stop()
    # samples that arrived while the timed steps ran (nvidia-smi prints each
    # shortly after taking it: a 25 ms allowance at the end)
    clocks = sampler.summary(t_begin, t_end + 0.025)
    roof_clocks = sampler.summary(t_rbegin, t_rend + 0.025)

    # ---- plan of the timed call: which kernels ran
    st, plan = sg.sgemm_plan_detail(w.transA, w.transB, w.M, w.N, w.K, lda, ldb, ldc, True, True,
                                    True, sg.PATH_AUTO, 0, sms)

    # ---- peaks
    peaks, peak_src = measured_peaks()
    max_mhz = clocks["sm_max_mhz"] or peaks.get("sm_max_mhz", 2070.0)
    med_mhz = clocks["sm_mhz"] or max_mhz
    roof_mhz = roof_clocks["sm_mhz"] or med_mhz
    ffma_peak = sms * FP32_LANES_PER_SM * 2 * max_mhz * 1e6 / 1e12
    ffma_peak_med = sms * FP32_LANES_PER_SM * 2 * med_mhz * 1e6 / 1e12
    # TF32 tensor peak, the recipe's rule: measured bf16 (burst) x nominal
    # tf32/bf16 ratio (1.1/2.25); and from the tensor pipe's measured
    # kind::tf32 rate (library probe) x SMs x 2 flop x SM clock
    tf32_peak = peaks["bf16_tflops"] * (1.1 / 2.25)
    pst, mac_rate = sg.sgemm_probe_tf32_rate(4096)
    if pst != 0:
        mac_rate = None
    tf32_rate_peak = (lambda mhz: sms * mac_rate * 2 * mhz * 1e6 / 1e12) if mac_rate else None

    # ---- per-path timings on the same workload (outside the timed region)
    paths = {}
    rows_s, cols_s = gi.sample_points(w.M, w.N, 2048, seed=w.seed)
    ref = bound = None
    if rank == 0 and not args.no_check:
        import oracle
        ref, bound = oracle.gemm_f64(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A, lda, B, ldb,
                                     w.beta, C, ldc, points=(rows_s, cols_s))
    wanted = set(args.paths.split(","))
    # The per-path timings start from an idle GPU (the power-capped clock of the
    # tensor-core steps above does not carry over into them), and each records
    # the SM clock samples taken while it ran.
    path_clocks = ClockSampler(local)
    path_clocks.start()
    time.sleep(1.0)
    for name, pid in (("ffma", sg.PATH_FFMA), ("3xtf32", sg.PATH_3XTF32), ("tf32", sg.PATH_TF32)):
        if name not in wanted:
            continue
        try:
            call(pid)
        except sg.SgemmError as e:
            paths[name] = {"status": e.status, "note": sg.sgemm_status_string(e.status)}
            continue
        torch.cuda.synchronize(dev)
        t_pb = time.perf_counter()
        ms = event_times(lambda: call(pid), stream, flush,
                         max(20 if name == "ffma" else 3, args.path_reps), True)
        t_pe = time.perf_counter()
        warm = event_times(lambda: call(pid), stream, flush, 5, False)
        t = statistics.median(ms)
        tfl = w.flops / (t / 1e3) / 1e12
        ent = {"ms": t, "ms_min": min(ms), "ms_unflushed": statistics.median(warm), "tflops": tfl}
        time.sleep(0.05)
        ck = path_clocks.summary(t_pb, t_pe + 0.025) if path_clocks.proc else path_clocks.summary()
        ent["clocks"] = {"sm_mhz": ck["sm_mhz"], "reasons": ck["reasons"], "samples": ck["samples"]}
        if name == "ffma":
            ent["frac_ffma_peak_max_clock"] = tfl / ffma_peak
            ent["frac_ffma_peak_median_clock"] = tfl / ffma_peak_med
            if ck["sm_mhz"]:
                ent["frac_ffma_peak_sampled_clock"] = tfl / (sms * FP32_LANES_PER_SM * 2 * ck["sm_mhz"] * 1e6 / 1e12)
        else:
            mult = 3 if name == "3xtf32" else 1
            ent["tensor_tflops"] = mult * tfl
            ent["frac_tf32_tensor_peak"] = mult * tfl / tf32_peak
            if tf32_rate_peak:
                ent["frac_tf32_rate_peak_max_clock"] = mult * tfl / tf32_rate_peak(max_mhz)
                if ck["sm_mhz"]:
                    ent["frac_tf32_rate_peak_sampled_clock"] = mult * tfl / tf32_rate_peak(ck["sm_mhz"])
        if ref is not None:
            import oracle
            out = dC.cpu().numpy()[rows_s, cols_s]
            rep = oracle.compare(out, ref, bound, w.K, w.alpha)
            ent.update({"oracle_pass": rep["pass"], "max_err_over_bound": rep["max_err_over_bound"],
                        "max_rel": rep["max_rel"]})
        paths[name] = ent
    path_clocks.stop()

    # ---- every workload through the selector, against its path's roofline
    workloads = None
    if rank == 0 and not args.no_workloads:
        workloads = workload_table(dev, stream, flush, ffma_peak, tf32_peak, peaks["hbm_gbs"],
                                   oracle_s=0.0 if (args.no_cpu or world > 1) else args.workload_oracle_s)

    # ---- dominant kernel of the timed call, from the roofline region
    main_name = {sg.PATH_FFMA: "ffma", sg.PATH_3XTF32: "3xtf32", sg.PATH_TF32: "tf32",
                 sg.PATH_GEMV: "gemv"}[plan["path"]]
    k_ms = statistics.mean(kernel_ms) if kernel_ms else ms_per_step
    mult = 3 if main_name == "3xtf32" else 1
    achieved = w.flops / (k_ms / 1e3) / 1e12          # useful flop rate of the kernel
    if main_name == "ffma":
        roofline = {"bound": "alu", "achieved": achieved, "peak": ffma_peak, "unit": "TFLOP/s",
                    "frac": achieved / ffma_peak,
                    "peak_median_clock": ffma_peak_med, "frac_median_clock": achieved / ffma_peak_med,
                    "peak_basis": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x "
                                  f"{max_mhz:.0f} MHz max SM clock (median under load {med_mhz:.0f} MHz)",
                    "kernel": "ffma_gemm_kernel"}
    else:
        tt = mult * achieved                           # tensor-pipe flop rate
        roofline = {"bound": "tensor", "achieved": tt, "peak": tf32_peak, "unit": "TFLOP/s",
                    "frac": tt / tf32_peak,
                    "peak_basis": f"{peak_src} bf16 {peaks['bf16_tflops']} TFLOP/s x 1.1/2.25 "
                                  "(nominal tf32/bf16 ratio)",
                    "kernel": "tc_gemm_kernel"}
        if tf32_rate_peak:
            roofline.update({
                "tf32_mac_per_clock_per_sm": mac_rate,
                "peak_tf32_rate_sampled_clock": tf32_rate_peak(roof_mhz),
                "frac_tf32_rate_sampled_clock": tt / tf32_rate_peak(roof_mhz),
                "peak_tf32_rate_max_clock": tf32_rate_peak(max_mhz),
                "frac_tf32_rate_max_clock": tt / tf32_rate_peak(max_mhz),
                "tf32_rate_basis": f"{sms} SMs x {mac_rate:.0f} MAC/clock/SM (measured, "
                                   "tcgen05.mma kind::tf32 128x256x8 issue loop) x 2 flop x SM "
                                   f"clock ({roof_mhz:.0f} MHz median in the roofline region; "
                                   f"{max_mhz:.0f} MHz max)"})
    roofline["traffic"] = traffic_from_profiles(roofline["kernel"] + ":" + w.name)
    roofline["kernel_ms"] = k_ms
    roofline["kernel_launches_timed"] = len(kernel_ms)
    roofline["timing"] = ("library CUDA event pair around each main-kernel launch, on the "
                          "launching stream, over a second region of the same steps")
    roofline["call_ms_with_events"] = statistics.mean(hooked_ms)
    if main_name != "ffma":
        roofline["useful_tflops"] = achieved

    # ---- end to end: the host-buffer entry point (pinned buffers); its copies
    # and the GEMM, pipelined by the library, are inside the timed region
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()
    if C is not None:
        hC.copy_(torch.from_numpy(C))

    def host_call():
        st = sg.sgemm_host(w.transA, w.transB, w.M, w.N, w.K, w.alpha, hA.data_ptr(), lda,
                           hB.data_ptr(), ldb, w.beta, hC.data_ptr(), ldc, stream)
        if st != 0:
            raise sg.SgemmError(st)

    for _ in range(2):
        host_call()
    barrier()
    e_steps = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(e_steps):
        host_call()
    torch.cuda.synchronize(dev)
    e_dt = time.perf_counter() - t0
    e2e_val = world * e_steps * w.flops / e_dt / 1e12
    h2d = A.nbytes + B.nbytes + (C.nbytes if C is not None else 0)
    d2h = w.M * w.N * 4
    e2e = {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "entry_point": "sgemm_host"}
    if ref is not None and w.beta == 0:
        import oracle
        rep = oracle.compare(hC.numpy()[rows_s, cols_s], ref, bound, w.K, w.alpha)
        e2e.update({"oracle_pass": rep["pass"], "max_err_over_bound": rep["max_err_over_bound"],
                    "oracle_points": int(rows_s.size)})

    # ---- CPU oracle baseline (rank 0, N == 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, rows, dt, threads = oracle_sample(w, A, B, C, seconds_target=args.ref_seconds)
        cpu = {"value": v / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"rows 0..{rows - 1} of C ({rows} x {w.N} outputs, "
                         f"{2 * rows * w.N * w.K:.3e} flop), {dt:.1f} s",
               "cpu_model": cpu_model()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "ms_per_step_min": min(step_ms),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(w),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches,
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                       "reasons": clocks["reasons"], "samples": clocks["samples"]},
            "roofline_clocks": {"sm_mhz": roof_clocks["sm_mhz"], "reasons": roof_clocks["reasons"],
                                "samples": roof_clocks["samples"]},
            "plan": plan, "paths": paths, "workloads": workloads, "ffma_peak_tflops": ffma_peak,
            "wall_s_timed": t_wall, "peaks_source": peak_src,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def only_path(args):
    """Profiling mode: W + K calls of one path on the workload, nothing else."""
    import torch
    import dense_fp32_gemm_05_gb300 as sg
    from dense_fp32_gemm_05_gb300 import build as sgbuild

    sgbuild.build()
    sg.load()
    w = gi.WORKLOADS[args.workload or WORKLOAD]
    A, B, C = gi.make_inputs(w)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = (torch.from_numpy(C).cuda() if C is not None
          else torch.empty((w.M, w.N), dtype=torch.float32, device="cuda"))
    pid = {"auto": sg.PATH_AUTO, "ffma": sg.PATH_FFMA, "3xtf32": sg.PATH_3XTF32,
           "tf32": sg.PATH_TF32}[args.only_path]
    s = torch.cuda.current_stream()
    ev = []
    for i in range(args.warmup + args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        st = sg.sgemm_ex(w.transA, w.transB, w.M, w.N, w.K, w.alpha, dA.data_ptr(), A.shape[1],
                         dB.data_ptr(), B.shape[1], w.beta, dC.data_ptr(), w.N, s, pid, 0)
        e1.record(s)
        if st != 0:
            raise sg.SgemmError(st)
        if i >= args.warmup:
            ev.append((e0, e1))
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev) if ev else None
    print(json.dumps({"mode": "only-path", "path": args.only_path, "workload": w.name,
                      "calls": args.warmup + args.steps, "median_ms": ms,
                      "tflops": (w.flops / ms / 1e9) if ms else None}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--path-reps", type=int, default=10)
    ap.add_argument("--ref-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--paths", default="ffma,3xtf32,tf32",
                    help="comma list of paths to time beside the main call")
    ap.add_argument("--only-path", default=None, choices=["auto", "ffma", "3xtf32", "tf32"],
                    help="profiling mode: run only W + K calls of this path on the "
                         "workload (no baseline, e2e or oracle) and print their timing")
    ap.add_argument("--workload", default=None, choices=list(gi.WORKLOADS),
                    help="profiling mode: the workload (default: the benchmark's)")
    ap.add_argument("--no-check", action="store_true", help="skip the oracle sample check")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload table (every workload through sgemm)")
    ap.add_argument("--workload-oracle-s", type=float, default=1.0,
                    help="seconds of CPU oracle time per workload in the table (0: none)")
    args = ap.parse_args()
    if args.impl == "reference":
        return reference_arm(args)
    if args.only_path:
        return only_path(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
