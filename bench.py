"""Benchmark: FP32 SGEMM GFLOP/s on one GB300 (and % of the FP32 FFMA peak).

One step = one C = alpha*A*B + beta*C call of the workload (default: the
4096^3 square problem, A,B ~ U[-1,1], seed 1, alpha 1, beta 0) through the
library's C ABI, inputs already resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--config VARIANT] [--kernel-only]

Timing: W >= 3 untimed warm-up steps, then K steps; before every step a
256 MiB buffer is written to flush the 129 MB L2 and then read back, so
that L2 holds neither the inputs nor dirty lines whose write-back would
land inside the step, outside that step's CUDA event pair on the launching
stream.  ms_per_step is the mean event time (the "workloads" records rate
each configuration by the median step instead, since a single host-side
stall among thousands of microsecond steps moves a mean of them);
under torchrun the max over ranks (each rank runs its own independent
problem: weak scaling, no collective on the data path).

Also reported: the end-to-end rate through sgemm_run_host (pinned host
buffers, H2D + kernel + D2H every step), cuBLAS SGEMM via torch.matmul with
TF32 off (context), the SM clock sampled with nvidia-smi during the timed
steps, the FFMA-peak fraction at that clock, and the CPU oracle timed on a
bounded sample on this host's cores.

"sustained": the headline workload run back to back for seconds, three
rounds, each reported as the median of its last three quarters with its SM
clock samples binned by MHz ("Writing a Fast Matmul in CUDA, Step by Step",
Step 1: warm up, time launches for seconds, keep the median, sample the
clock).  "workloads": every other workload (128^3, 4092^3 with alpha 0.5
and beta 3, the MLP shape, the 16- and 1-row decode shapes) through the
table's plan, each with its kernel time, roofline, ncu traffic, plan,
cuBLAS on the same inputs and the CPU oracle (in full, or the MLP shape's
first 1024 rows, extrapolated).

--impl reference times the fp64 CPU oracle (the reference arm) on the same
workload, one bounded row-band per step.
"""
from __future__ import annotations

import argparse
import datetime
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

METRIC = "FP32 SGEMM GFLOP/s at 4096^3 on 1 GB300; % of FP32 FFMA peak"
FMA_LANES_PER_SM = 128          # FP32 lanes per SM (4 sub-partitions x 32)
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
# The sources a variant family's kernel is built from: a traffic figure in
# profiles/traffic.json stays valid while their hash is unchanged.
KERNEL_SOURCES = {
    "tmat_64x": ["tmat_kernel.cuh", "tmat_variants_rows.cu", "tile_order.cuh", "ptx.cuh", "kernels.h"],
    "tmat_": ["tmat_kernel.cuh", "tmat_variants.cu", "tile_order.cuh", "ptx.cuh", "kernels.h"],
    "skinny": ["kernel_skinny.cu", "ptx.cuh", "kernels.h"],
    "tma_": ["tma_kernel.cuh", "tma_variants_a.cu", "tma_variants_b.cu", "tma_variants_c.cu", "tile_order.cuh", "ptx.cuh",
             "kernels.h"],
    "cpa_": ["cpa_kernel.cuh", "cpa_variants.cu", "tile_order.cuh", "ptx.cuh", "kernels.h"],
    "tf32x3": ["tc_tf32x3.cu", "ptx.cuh", "kernels.h"],
    "generic": ["kernel_generic.cu", "kernels.h"],
    "gemv": ["kernel_gemv.cu", "kernel_gemv.h", "kernels.h"],
    "tiny_": ["kernel_tiny.cu", "kernels.h"],
}


def kernel_source_hash(variant: str) -> str:
    """Hash of the sources of `variant`'s kernel family (all kernel sources for an unknown family)."""
    names = next((v for k, v in KERNEL_SOURCES.items() if variant.startswith(k)),
                 sorted({n for v in KERNEL_SOURCES.values() for n in v}))
    h = hashlib.sha256()
    for name in names:
        p = os.path.join(ROOT, "dense_fp32_matrix_sm_gb300", "csrc", name)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str, period_ms: int = 100):
        self.gpu_id = gpu_id
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        cmd = ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", str(self.period_ms)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.3)

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if not self.proc:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)

    def rows(self):
        """Parsed samples: host wall-clock time t (seconds), SM and max MHz, power, reasons."""
        out = []
        for ln in list(self.lines):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                out.append({"t": t, "sm": float(parts[1]), "max": float(parts[2]),
                            "power": float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else None,
                            "active": parts[4], "hw": parts[5], "hwt": parts[6], "swt": parts[7],
                            "swp": parts[8]})
            except ValueError:
                continue
        return out

    def summary(self, window=None):
        """Median SM clock and throttle reasons over every sample, or over the
        samples inside window = (t0, t1) (host wall-clock seconds)."""
        rows = self.rows()
        if window is not None:
            rows = [r for r in rows if window[0] <= r["t"] <= window[1]]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        sm = [r["sm"] for r in rows]
        powers = [r["power"] for r in rows if r["power"] is not None]
        bins = {}
        for v in sm:
            bins[str(int(v))] = bins.get(str(int(v)), 0) + 1
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r["max"] for r in rows),
                "sm_mhz_min": min(sm), "power_w_max": max(powers) if powers else None,
                "reasons": sorted(reasons), "samples": len(rows), "sm_mhz_bins": bins}


def gpu_id_for(torch, dev: int) -> str:
    props = torch.cuda.get_device_properties(dev)
    bus = getattr(props, "pci_bus_id", None)
    dom = getattr(props, "pci_domain_id", None)
    pdev = getattr(props, "pci_device_id", None)
    if bus is not None and dom is not None and pdev is not None:
        return f"{dom:08X}:{bus:02X}:{pdev:02X}.0"
    return str(dev)


# ---------------------------------------------------------------- CPU oracle

def time_oracle_rows(A, B, C0, w, rows: int, threads: int) -> float:
    import oracle

    Cs = C0[:rows] if w.beta != 0.0 else None
    t0 = time.perf_counter()
    oracle.sgemm_ref(A[:rows], B, Cs, w.alpha, w.beta, threads=threads)
    return time.perf_counter() - t0


def size_oracle_sample(A, B, C0, w, threads: int, target_s: float) -> int:
    """Rows per sample so that one oracle call takes about target_s seconds."""
    probe = min(w.M, max(threads, 1))
    t = time_oracle_rows(A, B, C0, w, probe, threads)
    per_row = t / probe
    rows = int(target_s / max(per_row, 1e-9))
    rows = max(min(w.M, threads), min(w.M, rows))
    if rows > threads:
        rows = rows // threads * threads
    return max(1, min(w.M, rows))


# ---------------------------------------------------------------- main

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="square4096")
    ap.add_argument("--config", default=None, help="force a kernel variant by name")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time only the library kernel (no e2e, cuBLAS or CPU legs)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="size of the CPU-baseline sample")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the record of the other workloads (kernel time, roofline, cuBLAS, CPU oracle)")
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="length of each round of the back-to-back leg (0: skip it)")
    return ap.parse_args()


def dist_setup(torch):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist, rank, world, local
    return None, rank, world, local


def max_over_ranks(torch, dist, value: float) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(torch, dist):
    if dist is not None:
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def run_reference(args):
    """The reference arm: the fp64 CPU oracle on bounded row-band samples."""
    import torch

    dist, rank, world, _ = dist_setup(torch)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    import oracle
    from dense_fp32_matrix_sm_gb300.inputs import WORKLOADS, workload_inputs

    oracle.build()
    w = WORKLOADS[args.workload]
    A, B, C0 = workload_inputs(w)
    threads = host_cores()
    total_steps = max(1, args.steps + args.warmup)
    per_step = max(0.05, min(5.0, 120.0 / total_steps))
    rows = size_oracle_sample(A, B, C0, w, threads, per_step)
    for _ in range(args.warmup):
        time_oracle_rows(A, B, C0, w, rows, threads)
    times = [time_oracle_rows(A, B, C0, w, rows, threads) for _ in range(max(1, args.steps))]
    t = sum(times) / len(times)
    flops = 2.0 * rows * w.N * w.K
    gflops = flops / t / 1e9
    sample = f"rows 0..{rows - 1} of {w.M} (all {w.N} columns, K={w.K}) per step"
    out = {
        "impl": "reference", "metric": METRIC, "value": round(gflops, 3), "unit": "GFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{w.name}: {w.describe()}", "M": w.M, "N": w.N, "K": w.K},
        "cpu_baseline": {"value": round(gflops, 3), "unit": "GFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gflops, 3), "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def time_steps(torch, fn, steps: int, flush, stream):
    """Per-step CUDA-event times (ms) of fn() on `stream`, flushing L2 before each."""
    evs = []
    for _ in range(steps):
        flush()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        evs.append((s, e))
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def traffic_for(variant, workload: str):
    """DRAM bytes per launch of `variant` on `workload` from profiles/traffic.json,
    or None when there is no capture or the kernel's sources changed since."""
    if not variant or not os.path.exists(TRAFFIC_FILE):
        return None
    try:
        rec = json.load(open(TRAFFIC_FILE)).get(f"{variant}|{workload}")
    except (ValueError, OSError):
        return None
    if rec and rec.get("kernel_source_sha") == kernel_source_hash(str(variant)):
        return rec.get("dram_bytes_per_launch")
    return None


def roofline_for(w, ms: float, sms: int, sm_mhz: float, peaks: dict, traffic):
    """The roofline of one workload's step time `ms`.  The bound follows the
    arithmetic intensity: below the ridge (FFMA peak at sm_mhz over the
    measured HBM copy bandwidth) the kernel is bound by HBM, above it by the
    FP32 FFMA pipe (SMs x 128 lanes x 2 FLOP x clock)."""
    peak_tflops = sms * FMA_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    hbm_gbs = peaks.get("hbm_gbs") or FALLBACK_HBM_GBS
    hbm_basis = ("MEASURED_PEAKS.json hbm_gbs, STREAM-style copy, burst (of measured)" if peaks.get("hbm_gbs")
                 else "fallback 6.8 TB/s (of fallback)")
    intensity = w.flops / w.algorithmic_bytes()
    ridge = peak_tflops * 1e12 / (hbm_gbs * 1e9)
    if intensity < ridge:
        achieved_gbs = w.algorithmic_bytes() / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm_gbs, "unit": "GB/s",
                "frac": round(achieved_gbs / hbm_gbs, 4), "traffic": traffic, "peak_basis": hbm_basis,
                "algorithmic_bytes": w.algorithmic_bytes(),
                "intensity_flop_per_byte": round(intensity, 2), "ridge_flop_per_byte": round(ridge, 2)}
    achieved_tflops = w.flops / (ms * 1e-3) / 1e12
    return {"bound": "alu", "achieved": round(achieved_tflops, 3), "peak": round(peak_tflops, 3),
            "unit": "TFLOP/s", "frac": round(achieved_tflops / peak_tflops, 4), "traffic": traffic,
            "peak_basis": "SMs x 128 FP32 lanes x 2 FLOP x median SM clock sampled during the timed steps "
                          "(FFMA pipe; not a tensor-core path)",
            "algorithmic_bytes": w.algorithmic_bytes(),
            "intensity_flop_per_byte": round(intensity, 2), "ridge_flop_per_byte": round(ridge, 2)}


def median_last_three_quarters(times):
    """Median of the last three quarters of a run of step times (the first
    quarter is the warming part of a back-to-back run)."""
    n = len(times)
    return statistics.median(times[n // 4:] if n >= 4 else times)


def cublas_step_fn(torch, w, dA, dB, dC0, out):
    """torch.matmul / addmm in FP32 with TF32 off: cuBLAS SGEMM, context only."""
    torch.backends.cuda.matmul.allow_tf32 = False
    torch.backends.cudnn.allow_tf32 = False
    if w.beta == 0.0:
        return lambda: torch.matmul(dA, dB, out=out)
    return lambda: torch.addmm(dC0, dA, dB, beta=w.beta, alpha=w.alpha, out=out)


# The pages' own sizes for the oracle on the host cores: the 128^3, 4092^3
# and few-row problems in full; the MLP shape (962 GFLOP) on its first 1024
# rows, scaled to the whole product.
CPU_ROWS = {"mlp": 1024}


def workloads_leg(torch, sg, names, stream, flush, warmup, steps, sms, peaks, sampler, cpu: bool, threads: int,
                  min_seconds: float = 0.5):
    """Every other workload through the table's plan, timed like the headline
    (L2 flushed before each step, CUDA events on the launching stream), with
    its roofline, its ncu traffic, its plan, cuBLAS on the same inputs and the
    oracle on the host cores.  Returns (records, kernel launches)."""
    from dense_fp32_matrix_sm_gb300.inputs import WORKLOADS, workload_inputs

    recs = {}
    launches = 0
    for name in names:
        w = WORKLOADS[name]
        A, B, C0 = workload_inputs(w)
        dA = torch.from_numpy(A).cuda()
        dB = torch.from_numpy(B).cuda()
        dC0 = torch.from_numpy(C0).cuda()
        dC = dC0.clone()
        plan = sg.Plan(w.M, w.N, w.K)
        info = plan.info()

        def step():
            plan.run(w.alpha, dA, dB, w.beta, dC, stream)

        for _ in range(warmup):
            flush()
            step()
        torch.cuda.synchronize()
        # at least `steps` steps and at least min_seconds of them, so that the
        # 100 ms clock samples cover every workload's timed region
        t0 = time.time()
        times = []
        while len(times) < steps or time.time() - t0 < min_seconds:
            times += time_steps(torch, step, steps, flush, stream)
        t1 = time.time()
        if sg.device_status() != sg.SGEMM_OK:
            raise SystemExit(f"kernel status word set during the {name} steps (a wait timed out)")
        launches += plan.launches * (len(times) + warmup)
        ms = statistics.fmean(times)
        ms_med = statistics.median(times)
        clk = sampler.summary(window=(t0 - 0.05, t1 + 0.05)) if sampler else {}
        mhz = clk.get("sm_mhz") or peaks.get("sm_max_mhz") or 2070.0
        rec = {"workload": f"{w.name}: {w.describe()}", "ms_per_step": round(ms, 5),
               "ms_median": round(ms_med, 5), "ms_min": round(min(times), 5),
               "steps": len(times), "timed_seconds": round(t1 - t0, 2),
               "gflops": round(w.flops / (ms_med * 1e-3) / 1e9, 1), "rate_from": "median step",
               "roofline": roofline_for(w, ms_med, sms, mhz, peaks, traffic_for(info.get("variant"), w.name)),
               "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
               "plan": plan.describe(), "gpu_launches_per_step": plan.launches}
        plan.close()
        # cuBLAS on the same inputs (context)
        out = torch.empty_like(dC)
        cb = cublas_step_fn(torch, w, dA, dB, dC0, out)
        for _ in range(warmup):
            cb()
        cb_ms = statistics.median(time_steps(torch, cb, steps, flush, stream))
        rec["cublas_context"] = {"gflops": round(w.flops / (cb_ms * 1e-3) / 1e9, 1), "ms": round(cb_ms, 5),
                                 "call": "torch.matmul/addmm fp32, allow_tf32=False"}
        del dA, dB, dC0, dC, out
        torch.cuda.empty_cache()
        if cpu:
            import oracle

            rows = min(w.M, CPU_ROWS.get(name, w.M))
            t = time_oracle_rows(A, B, C0, w, rows, threads)
            rec["cpu_baseline"] = {
                "value": round(2.0 * rows * w.N * w.K / t / 1e9, 3), "unit": "GFLOP/s", "cores": threads,
                "kind": "oracle",
                "sample": (f"all {w.M} rows, fp64 with the |A||B| bound, {t:.2f} s" if rows == w.M else
                           f"rows 0..{rows - 1} of {w.M} (all {w.N} columns, K={w.K}), fp64 with the |A||B| "
                           f"bound, {t:.2f} s; extrapolated to the whole product: "
                           f"{t * w.M / rows:.1f} s")}
        recs[name] = rec
    return recs, launches


def sustained_leg(torch, step, flush, stream, w, seconds: float, rounds: int, sms, sampler):
    """The pages' timing protocol on the headline workload: back-to-back steps
    for `seconds` (L2 flushed before each, per-step CUDA events), the median of
    the last three quarters, `rounds` times; the SM clock samples of each
    round binned by MHz, so the rate can be read against the clock."""
    out = []
    for _ in range(rounds):
        evs = []
        t0 = time.time()
        while time.time() - t0 < seconds:
            for _ in range(50):
                flush()
                s = torch.cuda.Event(enable_timing=True)
                e = torch.cuda.Event(enable_timing=True)
                s.record(stream)
                step()
                e.record(stream)
                evs.append((s, e))
            evs[-1][1].synchronize()
        torch.cuda.synchronize()
        t1 = time.time()
        times = [s.elapsed_time(e) for s, e in evs]
        med = median_last_three_quarters(times)
        clk = sampler.summary(window=(t0, t1)) if sampler else {}
        mhz = clk.get("sm_mhz")
        rec = {"steps": len(times), "seconds": round(t1 - t0, 2), "ms_median_last_3q": round(med, 5),
               "gflops": round(w.flops / (med * 1e-3) / 1e9, 1),
               "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_mhz_min", "reasons", "samples", "sm_mhz_bins",
                                                  "power_w_max")}}
        if mhz:
            rec["pct_ffma_peak_at_round_clock"] = round(
                100.0 * w.flops / (med * 1e-3) / (sms * FMA_LANES_PER_SM * 2 * mhz * 1e6), 2)
        out.append(rec)
    meds = [r["ms_median_last_3q"] for r in out]
    return {"rounds": out, "ms_median_of_rounds": round(statistics.median(meds), 5),
            "spread_pct": round(100.0 * (max(meds) - min(meds)) / statistics.median(meds), 2),
            "gflops": round(w.flops / (statistics.median(meds) * 1e-3) / 1e9, 1),
            "protocol": f"{rounds} rounds of >= {seconds:g} s of back-to-back steps, L2 flushed before each, "
                        "per-step CUDA events, median of the last three quarters of each round"}


TC_VARIANT = "tf32x3p_128x128x32_s3"


def tf32_peak_tflops(torch, stream, n: int = 8192, reps: int = 10):
    """The TF32 tensor-core rate measured with cuBLAS on this GPU: the best of
    `reps` torch.matmul calls on n^3 float32 operands with TF32 allowed
    (2 n^3 / time).  The denominator of the split-TF32 leg's roofline, as
    MEASURED_PEAKS.json's cuBLAS bf16 figure is for bf16."""
    prev = torch.backends.cuda.matmul.allow_tf32
    try:
        torch.backends.cuda.matmul.allow_tf32 = True
        a = torch.randn(n, n, device="cuda")
        b = torch.randn(n, n, device="cuda")
        c = torch.empty(n, n, device="cuda")
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = None
        for _ in range(reps):
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            torch.matmul(a, b, out=c)
            s1.record(stream)
            s1.synchronize()
            t = s0.elapsed_time(s1)
            best = t if best is None or t < best else best
        del a, b, c
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except RuntimeError:
        return None
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense tensor rates, TF32 over BF16


def tc_leg(torch, sg, w, dA, dB, dC0, stream, flush, warmup, steps, dist, peaks):
    """Time the split-TF32 variant like the main leg (L2 flushed, CUDA events) and
    report its agreement with the FFMA kernel on one fresh product."""
    plan = sg.Plan(w.M, w.N, w.K, config=TC_VARIANT)
    launches = plan.launches
    tC = dC0.clone()

    def tc_step():
        plan.run(w.alpha, dA, dB, w.beta, tC, stream)

    for _ in range(warmup):
        flush()
        tc_step()
    torch.cuda.synchronize()
    times = time_steps(torch, tc_step, steps, flush, stream)
    if sg.device_status() != sg.SGEMM_OK:
        raise SystemExit("kernel status word set during the split-TF32 steps")
    ms = max_over_ranks(torch, dist, statistics.fmean(times))
    # one fresh product from each path, compared elementwise
    c_tc = dC0.clone()
    plan.run(w.alpha, dA, dB, w.beta, c_tc, stream)
    ffma = sg.Plan(w.M, w.N, w.K)
    c_ff = dC0.clone()
    ffma.run(w.alpha, dA, dB, w.beta, c_ff, stream)
    torch.cuda.synchronize()
    rel = float(((c_tc - c_ff).abs().max() / c_ff.abs().max().clamp_min(1e-30)).item())
    ffma.close()
    desc = plan.describe()
    plan.close()
    bf16 = peaks.get("bf16_tflops")
    derived = round((bf16 if bf16 else 1900.0) * TF32_PER_BF16, 1)
    measured = tf32_peak_tflops(torch, stream)
    peak = round(measured, 1) if measured else derived
    tensor_tflops = 3 * w.flops / (ms * 1e-3) / 1e12  # three TF32 products per FP32 multiply-add
    return {"variant": TC_VARIANT, "value": round(w.flops / (ms * 1e-3) / 1e9, 1), "unit": "GFLOP/s",
            "ms_per_step": round(ms, 4), "steps": steps, "gpu_launches": launches * steps,
            "k_order": "tf32x3", "max_abs_diff_vs_ffma_rel_to_max_abs_c": rel,
            "roofline": {"bound": "tensor", "achieved": round(tensor_tflops, 1), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(tensor_tflops / peak, 4), "traffic": None,
                         "peak_basis": ("cuBLAS TF32 GEMM measured in this run: torch.matmul 8192^3 with allow_tf32, "
                                        "best of 10, CUDA events (of measured)" if measured else
                                        "MEASURED_PEAKS.json bf16_tflops (burst) x nominal TF32/BF16 ratio 1.1/2.25 "
                                        "(of measured)" if bf16 else "fallback 1.9 PF bf16 x 1.1/2.25 (of fallback)"),
                         "peak_derived_from_bf16": derived,
                         "achieved_basis": "3 x 2MNK TF32 tensor FLOPs over the whole step (the two split kernels "
                                           "included)"},
            "plan": desc}


def run_ours(args):
    import numpy as np
    import torch

    dist, rank, world, local = dist_setup(torch)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.cuda.current_device()
    from dense_fp32_matrix_sm_gb300 import build as b

    b.build()
    import dense_fp32_matrix_sm_gb300 as sg
    from dense_fp32_matrix_sm_gb300.inputs import WORKLOADS, workload_inputs

    w = WORKLOADS[args.workload]
    warmup = max(3, args.warmup)
    steps = max(1, args.steps)
    A, B, C0 = workload_inputs(w)
    dA = torch.from_numpy(A).to(dev)
    dB = torch.from_numpy(B).to(dev)
    dC0 = torch.from_numpy(C0).to(dev)
    dC = dC0.clone()
    flush_buf = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)   # 256 MiB > 129 MB L2
    stream = torch.cuda.current_stream()

    plan = sg.Plan(w.M, w.N, w.K, config=args.config)
    info = plan.info()
    launches_per_step = plan.launches

    def step():
        plan.run(w.alpha, dA, dB, w.beta, dC, stream)

    flush_sum = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        # write (evicts everything), then read (the written lines are clean
        # again, so their write-back is not charged to the next step)
        flush_buf.zero_()
        torch.sum(flush_buf, dim=0, out=flush_sum)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()

    sampler = None
    if rank == 0:
        sampler = ClockSampler(gpu_id_for(torch, dev))
        sampler.start()
    barrier(torch, dist)
    times = time_steps(torch, step, steps, flush, stream)
    barrier(torch, dist)
    if sampler:
        sampler.stop()
    if sg.device_status() != sg.SGEMM_OK:
        raise SystemExit("kernel status word set during the timed steps (a wait timed out)")

    ms = statistics.fmean(times)
    ms_max = max_over_ranks(torch, dist, ms)
    gflops_total = world * w.flops / (ms_max * 1e-3) / 1e9
    clocks = sampler.summary() if sampler else {}

    # the FP32 FFMA peak at the clock measured during the timed steps
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks = json.load(open(PEAKS_FILE)) if os.path.exists(PEAKS_FILE) else {}
    sm_mhz = clocks.get("sm_mhz") or None
    sm_max = clocks.get("sm_max_mhz") or peaks.get("sm_max_mhz") or 2070.0
    peak_tflops = sms * FMA_LANES_PER_SM * 2 * (sm_mhz or sm_max) * 1e6 / 1e12
    peak_max_tflops = sms * FMA_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    achieved_tflops = w.flops / (ms * 1e-3) / 1e12

    out = {
        "metric": METRIC, "value": round(gflops_total, 1), "unit": "GFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.describe()}", "M": w.M, "N": w.N, "K": w.K,
                   "variant": info.get("variant"), "grid": info.get("grid"),
                   "l2": "flushed before every timed step, outside its event pair: a 256 MiB buffer (> 129 MB L2) "
                         "written, then read back so no dirty line of it is written back inside the step",
                   "parallelism": "replicas" if world > 1 else "single"},
        "pct_ffma_peak": round(100.0 * achieved_tflops / peak_tflops, 2),
        "ffma_peak": {"sms": sms, "lanes_per_sm": FMA_LANES_PER_SM, "sm_mhz": sm_mhz,
                      "tflops_at_measured_clock": round(peak_tflops, 2),
                      "tflops_at_max_clock": round(peak_max_tflops, 2)},
        "step_ms": {"mean": round(ms, 4), "median": round(statistics.median(times), 4),
                    "min": round(min(times), 4), "max": round(max(times), 4)},
        "gpu_launches": launches_per_step * steps,
    }

    out["roofline"] = roofline_for(w, ms, sms, sm_mhz or sm_max, peaks, traffic_for(info.get("variant"), w.name))
    out["clocks"] = {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "sm_mhz_min",
                                                 "power_w_max", "samples")}

    # The FMA-only probe (after the timed steps): the FFMA pipe's achievable
    # rate, and the SM clock read inside a kernel, beside the nominal peak.
    p2_tflops, p2_mhz = sg.probe_ffma(True)
    p1_tflops, _ = sg.probe_ffma(False)
    nominal_at_probe = sms * FMA_LANES_PER_SM * 2 * p2_mhz * 1e6 / 1e12
    out["ffma_probe"] = {"ffma2_tflops": round(p2_tflops, 2), "ffma_tflops": round(p1_tflops, 2),
                         "sm_mhz_in_kernel": round(p2_mhz, 1),
                         "nominal_tflops_at_that_clock": round(nominal_at_probe, 2),
                         "ffma2_frac_of_nominal": round(p2_tflops / nominal_at_probe, 4),
                         "call": "sgemm_probe_ffma: the FFMA kernels' accumulation pattern without loads (4 x 8 FFMA2 pairs; 8 x 8 FFMA), 2 x 256-thread CTAs per SM"}
    if out["roofline"]["bound"] == "alu":
        out["roofline"]["frac_of_ffma2_probe"] = round(achieved_tflops / p2_tflops, 4)
    out["gpu_launches"] += 4

    if args.sustained_seconds > 0 and rank == 0 and sampler is not None:
        sampler2 = ClockSampler(gpu_id_for(torch, dev))
        sampler2.start()
        out["sustained"] = sustained_leg(torch, step, flush, stream, w, args.sustained_seconds, 3, sms, sampler2)
        sampler2.stop()
        out["gpu_launches"] += launches_per_step * sum(r["steps"] for r in out["sustained"]["rounds"])
        if sg.device_status() != sg.SGEMM_OK:
            raise SystemExit("kernel status word set during the sustained steps")

    if not args.kernel_only:
        # End to end from pinned host memory, every step copying its inputs in
        # and its result out.  Headline: sgemm_run_host_pipelined, where one
        # step's copies run under another step's kernel (two device buffer
        # sets).  Also reported: sgemm_run_host, one step at a time.
        hA = torch.from_numpy(A).pin_memory()
        hB = torch.from_numpy(B).pin_memory()
        hC2 = [torch.from_numpy(C0.copy()).pin_memory() for _ in range(2)]  # results alternate, so no host races
        h2d = hA.numel() * 4 + hB.numel() * 4 + (hC2[0].numel() * 4 if w.beta != 0.0 else 0)
        d2h = hC2[0].numel() * 4
        dA2, dB2, dC2 = [dA, dA.clone()], [dB, dB.clone()], [dC, dC.clone()]
        e2e_steps = max(3, min(steps, 50))

        def pipelined(n):
            plan.run_host_pipelined(w.alpha, [hA] * n, [hB] * n, w.beta, [hC2[i & 1] for i in range(n)], dA2, dB2,
                                    dC2, stream)

        pipelined(3)
        torch.cuda.synchronize()
        barrier(torch, dist)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        pipelined(e2e_steps)
        ev1.record(stream)  # the stream reaches this once every result is in host memory
        torch.cuda.synchronize()
        barrier(torch, dist)
        e2e_ms = max_over_ranks(torch, dist, ev0.elapsed_time(ev1) / e2e_steps)
        out["e2e"] = {"value": round(world * w.flops / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GFLOP/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                      "steps": e2e_steps,
                      "path": "sgemm_run_host_pipelined: per step cudaMemcpy2DAsync H2D of A and B (and C when "
                              "beta != 0) on one copy stream, the kernel, D2H of C on another; two device buffer "
                              "sets so copies overlap other steps' kernels; one event pair over all steps"}
        out["gpu_launches"] += launches_per_step * e2e_steps

        def e2e_step():
            plan.run_host(w.alpha, hA, hB, w.beta, hC2[0], dA, dB, dC, stream)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e2e_times = time_steps(torch, e2e_step, e2e_steps, flush, stream)
        e2e_serial_ms = max_over_ranks(torch, dist, statistics.fmean(e2e_times))
        out["e2e_serial"] = {"value": round(world * w.flops / (e2e_serial_ms * 1e-3) / 1e9, 1), "unit": "GFLOP/s",
                             "ms_per_step": round(e2e_serial_ms, 3), "steps": e2e_steps,
                             "path": "sgemm_run_host, one step at a time (H2D, kernel, D2H on one stream), L2 "
                                     "flushed before each step"}
        out["gpu_launches"] += launches_per_step * e2e_steps

        # cuBLAS SGEMM as context (TF32 off: plain FP32 results)
        tC = torch.empty_like(dC)
        cublas_step = cublas_step_fn(torch, w, dA, dB, dC0, tC)
        for _ in range(warmup):
            cublas_step()
        cb = time_steps(torch, cublas_step, min(steps, 100), flush, stream)
        cb_ms = statistics.fmean(cb)
        out["cublas_context"] = {"gflops": round(w.flops / (cb_ms * 1e-3) / 1e9, 1), "ms": round(cb_ms, 4),
                                 "call": "torch.matmul/addmm fp32, allow_tf32=False",
                                 "float32_matmul_precision": torch.get_float32_matmul_precision()}

        # The split-TF32 tensor-core variant on the same workload, reported on
        # its own: never the FFMA figure above.
        if TC_VARIANT in sg.config_names() and w.K >= 16:
            out["tf32x3"] = tc_leg(torch, sg, w, dA, dB, dC0, stream, flush, warmup, min(steps, 100), dist, peaks)

        if not args.no_workloads and rank == 0:
            from dense_fp32_matrix_sm_gb300.inputs import WORKLOADS

            names = [n for n in WORKLOADS if n != w.name]
            if world == 1:
                import oracle

                oracle.build()
            sampler3 = ClockSampler(gpu_id_for(torch, dev))
            sampler3.start()
            recs, n_launch = workloads_leg(torch, sg, names, stream, flush, warmup, max(20, min(steps, 50)), sms,
                                           peaks, sampler3, world == 1, host_cores())
            sampler3.stop()
            out["workloads"] = recs
            out["gpu_launches"] += n_launch

        if rank == 0 and world == 1:
            import oracle

            oracle.build()
            threads = host_cores()
            rows = size_oracle_sample(A, B, C0, w, threads, args.cpu_seconds)
            t = time_oracle_rows(A, B, C0, w, rows, threads)
            out["cpu_baseline"] = {"value": round(2.0 * rows * w.N * w.K / t / 1e9, 3), "unit": "GFLOP/s",
                                   "cores": threads, "kind": "oracle",
                                   "sample": f"rows 0..{rows - 1} of {w.M} (all {w.N} columns, K={w.K}), "
                                             f"fp64 with the |A||B| bound, {t:.1f} s"}
    out["plan"] = plan.describe()
    plan.close()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
