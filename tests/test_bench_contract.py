"""CPU checks of bench.py's contract pieces that need no GPU: the algorithmic
byte count of the headline workload, the lookup of committed DRAM traffic by
kernel tag and source hash, and the reference arm's JSON line (the CPU oracle
timed on a bounded sample)."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_of_the_headline():
    # N*M*4 bytes in + N*k*(4 + 4) bytes of CBSR out, N = 2^20, M = 256, k = 32
    assert bench.algorithmic_bytes(1 << 20, 256, 32, 4, 4, 4) == 1_342_177_280
    # MaxK forward (bf16 in, bf16 values, int16 indices)
    assert bench.algorithmic_bytes(1 << 20, 256, 32, 2, 2, 2) == 671_088_640


def test_profiled_traffic_needs_the_matching_source_hash():
    tag = "rtopk_select_f32_M256_k32"
    traffic, path = bench.profiled_traffic(tag, "0000000000000000")
    assert traffic is None and path is not None  # a profile exists, but not for these sources
    _, path2 = bench.profiled_traffic("no_such_kernel_tag", bench.kernel_source_hash())
    assert path2 is None


def test_reference_arm_prints_one_json_line():
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                        "--ref-seconds", "4"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads(p.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "rows/s" and line["value"] > 0
    assert line["higher_is_better"] is True and line["steps"] == 1 and line["warmup"] >= 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    # the same workload keys as the GPU arm's line
    assert line["config"] == bench.workload_config(1)
    assert line["cpu_baseline"]["cpu_model"]
