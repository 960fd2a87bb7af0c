"""Measure every kernel variant on given shapes (the autotuning sweep behind
the per-shape config table).

"How a Matmul Kernel Gets Fast", section 12 "Kernel 9: autotuning": compile
the legal tile configurations, run each on the problem, keep the fastest.
Here every variant is already compiled into the library; this times each
one with CUDA events (L2 flushed before every launch) and prints one JSON
line per (shape, variant) plus the winner per shape.

  python -m dense_fp32_matrix_sm_gb300.sweep --shapes 4096x4096x4096,16x16384x8192 \
      [--variants name,name] [--iters 30] [--warmup 5]
"""
from __future__ import annotations

import argparse
import json
import statistics
import sys


def parse_shape(s: str):
    m, n, k = (int(x) for x in s.lower().split("x"))
    return m, n, k


def time_variant(sg, torch, M, N, K, name, iters, warmup, flush_buf, A, B, C, beta):
    try:
        plan = sg.Plan(M, N, K, config=name)
    except sg.SgemmError as e:
        return {"variant": name, "status": e.status, "error": str(e)}
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        plan.run(1.0, A, B, beta, C, stream)
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        flush_buf.zero_()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        plan.run(1.0, A, B, beta, C, stream)
        e.record(stream)
        times.append((s, e))
    torch.cuda.synchronize()
    ms = [s.elapsed_time(e) for s, e in times]
    status = sg.device_status()
    info = plan.info()
    plan.close()
    med = statistics.median(ms)
    return {"variant": name, "M": M, "N": N, "K": K, "ms_median": round(med, 4), "ms_min": round(min(ms), 4),
            "gflops": round(2.0 * M * N * K / (med * 1e-3) / 1e9, 1), "grid": info.get("grid"),
            "ctas_per_sm": info.get("ctas_per_sm"), "status": status}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--shapes", default="4096x4096x4096")
    ap.add_argument("--variants", default="")
    ap.add_argument("--iters", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--beta", type=float, default=0.0)
    args = ap.parse_args(argv)

    import torch

    import dense_fp32_matrix_sm_gb300 as sg
    from dense_fp32_matrix_sm_gb300.inputs import make_inputs

    names = [v for v in args.variants.split(",") if v] or sg.config_names()
    flush_buf = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")
    for shape in args.shapes.split(","):
        M, N, K = parse_shape(shape)
        A, B, C0 = make_inputs(M, N, K, seed=1)
        dA = torch.from_numpy(A).cuda()
        dB = torch.from_numpy(B).cuda()
        dC = torch.from_numpy(C0).cuda()
        results = []
        for name in names:
            r = time_variant(sg, torch, M, N, K, name, args.iters, args.warmup, flush_buf, dA, dB, dC, args.beta)
            results.append(r)
            print(json.dumps(r), flush=True)
        ok = [r for r in results if r.get("status") == 0 and "gflops" in r]
        if ok:
            best = max(ok, key=lambda r: r["gflops"])
            print(json.dumps({"shape": shape, "best": best["variant"], "gflops": best["gflops"]}), flush=True)
        del dA, dB, dC
        torch.cuda.empty_cache()
    return 0


if __name__ == "__main__":
    sys.exit(main())
