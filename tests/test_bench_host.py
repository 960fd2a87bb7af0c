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
        "2070, 2070, 500.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 700.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 650.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    sm = s.summary()
    assert sm["sm_mhz"] == 2070.0 and sm["sm_max_mhz"] == 2070.0 and sm["samples"] == 3
    assert sm["reasons"] == ["sw_power_cap"]
    assert sm["power_w_max"] == 700.5
    empty = bench.ClockSampler("0").summary()
    assert empty["sm_mhz"] is None and empty["samples"] == 0


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
