"""Host-side logic of bench.py that needs no GPU: the max-over-ranks timing
reduction on a 2-rank gloo group, the clock-sample parser, and the
reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(torch, dist, 1.5 + rank * 2.25)
    bench.barrier(torch, dist)
    with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
        f.write(repr(got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    vals = [float(open(tmp_path / f"r{r}").read()) for r in range(2)]
    assert vals == [3.75, 3.75]


def test_clock_sampler_summary():
    import bench

    s = bench.ClockSampler("0")
    s.lines = [
        "2026/12/02 10:00:00.100, 2070, 2070, 500.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.200, 1980, 2070, 700.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.300, 2070, 2070, 650.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    sm = s.summary()
    assert sm["sm_mhz"] == 2070.0 and sm["sm_max_mhz"] == 2070.0 and sm["samples"] == 3
    assert sm["reasons"] == ["sw_power_cap"]
    assert sm["power_w_max"] == 700.5
    assert sm["sm_mhz_bins"] == {"2070": 2, "1980": 1}
    # a window keeps only the samples taken inside it (host wall-clock seconds)
    import datetime
    t = datetime.datetime(2026, 12, 2, 10, 0, 0, 150000).timestamp()
    win = s.summary(window=(t, t + 0.1))
    assert win["samples"] == 1 and win["sm_mhz"] == 1980.0 and win["reasons"] == ["sw_power_cap"]
    empty = bench.ClockSampler("0").summary()
    assert empty["sm_mhz"] is None and empty["samples"] == 0


def test_last_three_quarters_median():
    import bench

    # the first quarter (warming) is dropped, the median of the rest kept
    assert bench.median_last_three_quarters([9.0, 9.0, 1.0, 2.0, 3.0, 4.0, 5.0, 6.0]) == 3.5
    assert bench.median_last_three_quarters([2.0]) == 2.0


def test_roofline_bound_follows_intensity():
    import bench
    from dense_fp32_matrix_sm_gb300.inputs import WORKLOADS

    peaks = {"hbm_gbs": 6783.1}
    # 4096^3: far right of the ridge, the FFMA pipe bounds it
    r = bench.roofline_for(WORKLOADS["square4096"], 2.0, 152, 2070.0, peaks, None)
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert abs(r["peak"] - 152 * 128 * 2 * 2070e6 / 1e12) < 1e-3
    assert abs(r["achieved"] - 2 * 4096 ** 3 / 2e-3 / 1e12) < 1e-3
    # 16 x 16384 x 8192: below the ridge, HBM bounds it; bytes A + B + 2C
    r = bench.roofline_for(WORKLOADS["decode16"], 0.1, 152, 2070.0, peaks, 123)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6783.1 and r["traffic"] == 123
    assert r["algorithmic_bytes"] == 4 * (16 * 8192 + 8192 * 16384 + 2 * 16 * 16384)
    assert abs(r["frac"] - r["algorithmic_bytes"] / 0.1e-3 / 1e9 / 6783.1) < 1e-4


def test_reference_arm_line():
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "square128", "--steps", "2",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["unit"] == "GFLOP/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["metric"].startswith("FP32 SGEMM GFLOP/s")
